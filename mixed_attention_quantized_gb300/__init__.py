"""Python binding of ``libmixattn.so``: the mixed-batch attention step over a
block-quantised paged KV cache, GB300 (sm_103a).

This module only marshals arguments (torch tensors -> device pointers, the
current CUDA stream) into the C ABI declared in ``include/mixattn.h``; every
step of the path runs in the library's CUDA kernels.  There is no CPU
fallback: if the library is missing or fails to load, every call raises.

Reference: page "自研RDNA高併發推論引擎 以AI Max+ 395為範例" (§1 mixed batch,
§2 blocked Q8 / 4-bit KV modes).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

F16, Q8_0, Q4_0 = 0, 1, 2
ROW_DECODE, ROW_CHUNK = 0, 1
PAGE = 32

OK = 0
ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_DEVICE_CHECK = -1, -2, -3, -4, -5
DEVERR_PAGE_ID, DEVERR_SLOT, DEVERR_TIMEOUT = 0x1, 0x2, 0x4

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmixattn.so")

EXPORTED = [
    "mixattn_kv_cache_bytes", "mixattn_kv_append_quant", "mixattn_kv_export_blocks",
    "mixattn_plan_create", "mixattn_plan_create_window", "mixattn_plan_update", "mixattn_plan_info", "mixattn_run",
    "mixattn_plan_destroy", "mixattn_mixed_attention", "mixattn_workspace_bytes",
    "mixattn_device_error", "mixattn_status_string", "mixattn_version",
    "mixattn_mixed_attention_noalloc",
    "mixattn_sched_default_config", "mixattn_sched_create", "mixattn_sched_destroy", "mixattn_sched_submit",
    "mixattn_sched_next_batch", "mixattn_sched_complete", "mixattn_sched_request_info", "mixattn_sched_counts",
]

ERR_CLIENT_QUOTA = -6
STEP_IDLE, STEP_DECODE, STEP_MERGED, STEP_PREFILL = 0, 1, 2, 3
REQ_WAITING, REQ_PREFILL, REQ_DECODE, REQ_DONE = 0, 1, 2, 3


class MixattnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class SchedConfig(ctypes.Structure):
    _fields_ = [
        ("max_sessions", ctypes.c_int32), ("prefill_chunk", ctypes.c_int32),
        ("max_pending_per_client", ctypes.c_int32), ("near_done_tokens", ctypes.c_int32),
        ("max_decode_rows", ctypes.c_int32),
    ]


class KVCacheDesc(ctypes.Structure):
    _fields_ = [
        ("num_pages", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("k_fmt", ctypes.c_int32), ("v_fmt", ctypes.c_int32),
        ("k_quant", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
        ("v_quant", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
    ]


_lib = None


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the library (building it first if it is absent or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if path is None:
        from . import build as _build
        path = _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"libmixattn.so not found at {path}")
    lib = ctypes.CDLL(path)
    i32, i64, sz, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p
    i32p = ctypes.POINTER(ctypes.c_int32)
    cachep = ctypes.POINTER(KVCacheDesc)
    lib.mixattn_kv_cache_bytes.argtypes = [cachep, ctypes.POINTER(sz)]
    lib.mixattn_kv_cache_bytes.restype = sz
    lib.mixattn_kv_append_quant.argtypes = [cachep, vp, vp, vp, i32, vp]
    lib.mixattn_kv_append_quant.restype = ctypes.c_int
    lib.mixattn_kv_export_blocks.argtypes = [cachep, i32, vp, i32, vp, vp]
    lib.mixattn_kv_export_blocks.restype = ctypes.c_int
    lib.mixattn_plan_create.argtypes = [ctypes.POINTER(vp), cachep, i32, i32, i32p, i32p, i32p, i32,
                                        ctypes.POINTER(sz)]
    lib.mixattn_plan_create.restype = ctypes.c_int
    lib.mixattn_plan_create_window.argtypes = [ctypes.POINTER(vp), cachep, i32, i32, i32, i32p, i32p, i32p, i32,
                                               ctypes.POINTER(sz)]
    lib.mixattn_plan_create_window.restype = ctypes.c_int
    lib.mixattn_plan_update.argtypes = [vp, i32, i32p, i32p, i32p, i32, ctypes.POINTER(sz)]
    lib.mixattn_plan_update.restype = ctypes.c_int
    lib.mixattn_plan_info.argtypes = [vp, i32p, i32p, i32p]
    lib.mixattn_plan_info.restype = ctypes.c_int
    lib.mixattn_run.argtypes = [vp, vp, vp, vp, vp, sz, vp]
    lib.mixattn_run.restype = ctypes.c_int
    lib.mixattn_plan_destroy.argtypes = [vp]
    lib.mixattn_plan_destroy.restype = None
    lib.mixattn_mixed_attention.argtypes = [cachep, i32, vp, vp, i32, i32, i32p, i32p, i32p, vp, vp, sz, vp]
    lib.mixattn_mixed_attention.restype = ctypes.c_int
    lib.mixattn_mixed_attention_noalloc.argtypes = [cachep, i32, vp, vp, i32, i32, i32p, i32p, i32p, vp, vp]
    lib.mixattn_mixed_attention_noalloc.restype = ctypes.c_int
    lib.mixattn_workspace_bytes.argtypes = [cachep, i32, i32, i32p, i32p, i32p, i32, ctypes.POINTER(sz)]
    lib.mixattn_workspace_bytes.restype = ctypes.c_int
    lib.mixattn_device_error.argtypes = [i32]
    lib.mixattn_device_error.restype = i64
    lib.mixattn_status_string.argtypes = [i32]
    lib.mixattn_status_string.restype = ctypes.c_char_p
    lib.mixattn_version.argtypes = []
    lib.mixattn_version.restype = i32
    cfgp = ctypes.POINTER(SchedConfig)
    i64p = ctypes.POINTER(ctypes.c_int64)
    lib.mixattn_sched_default_config.argtypes = [cfgp]
    lib.mixattn_sched_default_config.restype = None
    lib.mixattn_sched_create.argtypes = [ctypes.POINTER(vp), cfgp]
    lib.mixattn_sched_create.restype = ctypes.c_int
    lib.mixattn_sched_destroy.argtypes = [vp]
    lib.mixattn_sched_destroy.restype = None
    lib.mixattn_sched_submit.argtypes = [vp, i64, i32, i32, i32]
    lib.mixattn_sched_submit.restype = ctypes.c_int
    lib.mixattn_sched_next_batch.argtypes = [vp, i32, i32p, i32p, i32p, i64p, i32p]
    lib.mixattn_sched_next_batch.restype = i32
    lib.mixattn_sched_complete.argtypes = [vp, i64p, i32]
    lib.mixattn_sched_complete.restype = ctypes.c_int
    lib.mixattn_sched_request_info.argtypes = [vp, i64, i32p, i32p, i32p, i64p, i64p]
    lib.mixattn_sched_request_info.restype = ctypes.c_int
    lib.mixattn_sched_counts.argtypes = [vp, i32p, i32p, i32p, i64p]
    lib.mixattn_sched_counts.restype = ctypes.c_int
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().mixattn_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != OK:
        raise MixattnError(status, what)


def _i32_array(values: Sequence[int]):
    arr = (ctypes.c_int32 * len(values))(*[int(v) for v in values])
    return arr


def _stream_handle(stream) -> ctypes.c_void_p:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream))


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(int(t.data_ptr())) if t is not None else ctypes.c_void_p(0)


def block_bytes(fmt: int) -> int:
    return {F16: 64, Q8_0: 34, Q4_0: 18}[fmt]


def row_bytes(fmt: int, head_dim: int) -> int:
    return {F16: 2 * head_dim, Q8_0: head_dim, Q4_0: head_dim // 2}[fmt]


def cache_desc(num_pages: int, num_kv_heads: int, head_dim: int, k_fmt: int, v_fmt: int,
               k_quant=0, k_scale=0, v_quant=0, v_scale=0) -> KVCacheDesc:
    return KVCacheDesc(num_pages, PAGE, num_kv_heads, head_dim, k_fmt, v_fmt,
                       k_quant, k_scale, v_quant, v_scale)


def kv_cache_bytes(desc: KVCacheDesc):
    """(total, [k_quant, k_scale, v_quant, v_scale]) bytes; total 0 if invalid."""
    planes = (ctypes.c_size_t * 4)()
    total = load().mixattn_kv_cache_bytes(ctypes.byref(desc), planes)
    return int(total), [int(x) for x in planes]


@dataclass
class KVCache:
    """Device planes of a paged KV cache (torch owns the memory)."""
    num_pages: int
    num_kv_heads: int
    head_dim: int
    k_fmt: int
    v_fmt: int
    k_quant: "object" = None
    k_scale: "object" = None
    v_quant: "object" = None
    v_scale: "object" = None

    @classmethod
    def allocate(cls, num_pages: int, num_kv_heads: int, head_dim: int, k_fmt: int, v_fmt: int,
                 device="cuda", fill: Optional[int] = 0) -> "KVCache":
        import torch
        c = cls(num_pages, num_kv_heads, head_dim, k_fmt, v_fmt)
        _, planes = kv_cache_bytes(c.desc(raw=True))
        if sum(planes) == 0:
            raise MixattnError(ERR_INVALID_ARG, "KVCache.allocate")

        def plane(n):
            if n == 0:
                return None
            t = torch.empty(n + 256, dtype=torch.uint8, device=device)
            off = (-t.data_ptr()) % 256
            v = t[off:off + n]
            if fill is not None:
                v.fill_(fill)
            return v
        c.k_quant, c.k_scale, c.v_quant, c.v_scale = (plane(n) for n in planes)
        return c

    def desc(self, raw: bool = False) -> KVCacheDesc:
        if raw:
            return cache_desc(self.num_pages, self.num_kv_heads, self.head_dim, self.k_fmt, self.v_fmt)
        return cache_desc(self.num_pages, self.num_kv_heads, self.head_dim, self.k_fmt, self.v_fmt,
                          _ptr(self.k_quant), _ptr(self.k_scale), _ptr(self.v_quant), _ptr(self.v_scale))


def kv_append_quant(cache: KVCache, k_new, v_new, slot_mapping, stream=None) -> None:
    """Quantise fp16 K/V ``[n_new, Hkv, D]`` into the cache slots ``slot_mapping`` (int32)."""
    n = int(k_new.shape[0]) if k_new is not None else 0
    st = load().mixattn_kv_append_quant(ctypes.byref(cache.desc()), _ptr(k_new), _ptr(v_new),
                                        _ptr(slot_mapping), n, _stream_handle(stream))
    _check(st, "mixattn_kv_append_quant")


def kv_export_blocks(cache: KVCache, which: int, slots, stream=None):
    """Canonical blocks ``[n, Hkv, D/32, block_bytes]`` (uint8, device) of K (0) or V (1)."""
    import torch
    fmt = cache.k_fmt if which == 0 else cache.v_fmt
    n = int(slots.shape[0])
    out = torch.empty((n, cache.num_kv_heads, cache.head_dim // 32, block_bytes(fmt)),
                      dtype=torch.uint8, device=slots.device)
    st = load().mixattn_kv_export_blocks(ctypes.byref(cache.desc()), int(which), _ptr(slots), n,
                                         _ptr(out), _stream_handle(stream))
    _check(st, "mixattn_kv_export_blocks")
    return out


class Plan:
    """Host tiling of one ForwardBatch; reusable across layers and re-tileable.
    ``window`` > 0 makes every run sliding-window attention (keys p-window+1..p)."""

    def __init__(self, cache: KVCache, num_q_heads: int, row_kinds, seq_lens, q_offsets,
                 max_pages: int, window: int = 0):
        self._lib = load()
        self.cache = cache
        self.num_q_heads = int(num_q_heads)
        self.window = int(window)
        self._handle = ctypes.c_void_p(0)
        ws = ctypes.c_size_t(0)
        self._desc = cache.desc()
        n = len(seq_lens)
        st = self._lib.mixattn_plan_create_window(ctypes.byref(self._handle), ctypes.byref(self._desc),
                                                  self.num_q_heads, self.window, n, _i32_array(row_kinds),
                                                  _i32_array(seq_lens), _i32_array(q_offsets),
                                                  int(max_pages), ctypes.byref(ws))
        _check(st, "mixattn_plan_create")
        self.workspace_bytes = int(ws.value)

    def update(self, row_kinds, seq_lens, q_offsets, max_pages: int) -> None:
        ws = ctypes.c_size_t(0)
        st = self._lib.mixattn_plan_update(self._handle, len(seq_lens), _i32_array(row_kinds),
                                           _i32_array(seq_lens), _i32_array(q_offsets),
                                           int(max_pages), ctypes.byref(ws))
        _check(st, "mixattn_plan_update")
        self.workspace_bytes = int(ws.value)

    def info(self):
        tq, nc, nd = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        _check(self._lib.mixattn_plan_info(self._handle, ctypes.byref(tq), ctypes.byref(nc),
                                           ctypes.byref(nd)), "mixattn_plan_info")
        return {"total_q": tq.value, "chunk_tiles": nc.value, "decode_tiles": nd.value}

    def run(self, q, page_table, o, workspace, stream=None) -> None:
        st = self._lib.mixattn_run(self._handle, _ptr(q), _ptr(page_table), _ptr(o), _ptr(workspace),
                                   int(workspace.numel() * workspace.element_size()),
                                   _stream_handle(stream))
        _check(st, "mixattn_run")

    def close(self) -> None:
        if self._handle and self._handle.value:
            self._lib.mixattn_plan_destroy(self._handle)
            self._handle = ctypes.c_void_p(0)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def workspace_bytes(cache: KVCache, num_q_heads: int, row_kinds, seq_lens, q_offsets,
                    max_pages: int) -> int:
    ws = ctypes.c_size_t(0)
    st = load().mixattn_workspace_bytes(ctypes.byref(cache.desc(raw=True)), int(num_q_heads),
                                        len(seq_lens), _i32_array(row_kinds), _i32_array(seq_lens),
                                        _i32_array(q_offsets), int(max_pages), ctypes.byref(ws))
    _check(st, "mixattn_workspace_bytes")
    return int(ws.value)


def alloc_workspace(nbytes: int, device="cuda"):
    """A 256-byte aligned uint8 device buffer of nbytes (torch-owned)."""
    import torch
    t = torch.empty(nbytes + 256, dtype=torch.uint8, device=device)
    off = (-t.data_ptr()) % 256
    return t[off:off + nbytes]


def mixed_attention(cache: KVCache, q, page_table, seq_lens, q_offsets, row_kinds, o=None,
                    workspace=None, stream=None):
    """o = mixed_attention(q, page_table, seq_lens, q_offsets, row_kinds) in one call."""
    import torch
    max_pages = int(page_table.shape[1])
    hq = int(q.shape[1])
    need = workspace_bytes(cache, hq, row_kinds, seq_lens, q_offsets, max_pages)
    if workspace is None:
        workspace = alloc_workspace(need, q.device)
    if o is None:
        o = torch.empty_like(q)
    st = load().mixattn_mixed_attention(
        ctypes.byref(cache.desc()), hq, _ptr(q), _ptr(page_table), max_pages, len(seq_lens),
        _i32_array(seq_lens), _i32_array(q_offsets), _i32_array(row_kinds), _ptr(o), _ptr(workspace),
        int(workspace.numel()), _stream_handle(stream))
    _check(st, "mixattn_mixed_attention")
    return o


def mixed_attention_noalloc(cache: KVCache, q, page_table, seq_lens, q_offsets, row_kinds, o=None,
                            stream=None):
    """Same step with the workspace held by the library (nothing is allocated
    by the call): for callers that cannot provide device scratch memory.
    Batches needing more than the library's 16 MiB of scratch raise
    MixattnError(ERR_WORKSPACE); overlapping calls on different streams race."""
    import torch
    if o is None:
        o = torch.empty_like(q)
    st = load().mixattn_mixed_attention_noalloc(
        ctypes.byref(cache.desc()), int(q.shape[1]), _ptr(q), _ptr(page_table), int(page_table.shape[1]),
        len(seq_lens), _i32_array(seq_lens), _i32_array(q_offsets), _i32_array(row_kinds), _ptr(o),
        _stream_handle(stream))
    _check(st, "mixattn_mixed_attention_noalloc")
    return o


def device_error(clear: bool = False) -> int:
    v = int(load().mixattn_device_error(1 if clear else 0))
    if v < 0:
        raise MixattnError(v, "mixattn_device_error")
    return v


def version() -> int:
    return int(load().mixattn_version())


@dataclass
class Batch:
    """One step built by the fair batch builder: the attention ABI's row arrays."""
    kind: int
    row_kinds: list
    seq_lens: list
    q_offsets: list
    request_ids: list


class FairBatchBuilder:
    """The host fair batch builder (``include/mixattn_sched.h``): requests in,
    ForwardBatch row arrays out (decode first, one bounded prefill slice per
    step, SRTF, starvation preemption behind the near-done gate,
    MarkAllDecodersDue, PopDecoder rotation, per-client admission)."""

    def __init__(self, max_sessions: int = 16, prefill_chunk: int = 512, max_pending_per_client: int = 0,
                 near_done_tokens: int = 64, max_decode_rows: int = 0):
        self._lib = load()
        self.config = SchedConfig(max_sessions, prefill_chunk, max_pending_per_client, near_done_tokens,
                                  max_decode_rows)
        self._h = ctypes.c_void_p(0)
        _check(self._lib.mixattn_sched_create(ctypes.byref(self._h), ctypes.byref(self.config)),
               "mixattn_sched_create")
        cap = max_sessions + 1
        self._cap = cap
        self._kinds = (ctypes.c_int32 * cap)()
        self._seq = (ctypes.c_int32 * cap)()
        self._off = (ctypes.c_int32 * cap)()
        self._ids = (ctypes.c_int64 * cap)()

    @staticmethod
    def default_config() -> SchedConfig:
        c = SchedConfig()
        load().mixattn_sched_default_config(ctypes.byref(c))
        return c

    def submit(self, request_id: int, client_id: int, prompt_len: int, max_new_tokens: int) -> int:
        """Queue a request; returns OK or ERR_CLIENT_QUOTA (other statuses raise)."""
        st = self._lib.mixattn_sched_submit(self._h, int(request_id), int(client_id), int(prompt_len),
                                            int(max_new_tokens))
        if st not in (OK, ERR_CLIENT_QUOTA):
            _check(st, "mixattn_sched_submit")
        return st

    def next_batch(self) -> Batch:
        kind = ctypes.c_int32(0)
        n = self._lib.mixattn_sched_next_batch(self._h, self._cap, self._kinds, self._seq, self._off, self._ids,
                                               ctypes.byref(kind))
        if n < 0:
            _check(n, "mixattn_sched_next_batch")
        return Batch(kind.value, list(self._kinds[:n]), list(self._seq[:n]), list(self._off[:n]),
                     list(self._ids[:n]))

    def complete(self, stop_ids=()) -> None:
        ids = list(stop_ids)
        arr = (ctypes.c_int64 * max(1, len(ids)))(*ids)
        _check(self._lib.mixattn_sched_complete(self._h, arr, len(ids)), "mixattn_sched_complete")

    def info(self, request_id: int) -> dict:
        st, ca, ge = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        ft, dn = ctypes.c_int64(), ctypes.c_int64()
        _check(self._lib.mixattn_sched_request_info(self._h, int(request_id), ctypes.byref(st), ctypes.byref(ca),
                                                    ctypes.byref(ge), ctypes.byref(ft), ctypes.byref(dn)),
               "mixattn_sched_request_info")
        return {"state": st.value, "cached": ca.value, "generated": ge.value, "first_token_step": ft.value,
                "done_step": dn.value}

    def counts(self) -> dict:
        w, p, d = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        n = ctypes.c_int64()
        _check(self._lib.mixattn_sched_counts(self._h, ctypes.byref(w), ctypes.byref(p), ctypes.byref(d),
                                              ctypes.byref(n)), "mixattn_sched_counts")
        return {"waiting": w.value, "prefills": p.value, "decoders": d.value, "steps": n.value}

    def close(self) -> None:
        if self._h and self._h.value:
            self._lib.mixattn_sched_destroy(self._h)
            self._h = ctypes.c_void_p(0)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
