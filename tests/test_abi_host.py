"""Host-side checks of the C ABI (no GPU needed): the library builds and loads,
exports every function ``include/mixattn.h`` declares, sizes the cache per the
reference page's byte table, and rejects bad arguments before any launch."""
import ctypes
import json
import os
import re

import numpy as np
import pytest

import mixed_attention_quantized_gb300 as mq
import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 1 << 20  # 256-byte aligned non-null "device" address; never dereferenced on the host


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", fn)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(mixattn_\w+)\s*\(", src, flags=re.M):
            names.append(m.group(1))
    return sorted(set(names))


def test_library_exports_every_declared_function():
    lib = mq.load()
    declared = _declared_functions()
    assert len(declared) >= 13, declared
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    assert set(mq.EXPORTED) <= set(declared)


def test_version_and_status_strings():
    assert mq.version() == 100
    assert mq.status_string(mq.OK) == "ok"
    assert "workspace" in mq.status_string(mq.ERR_WORKSPACE)
    assert mq.status_string(12345) == "unknown status"


def test_cache_bytes_reproduce_the_occupancy_table(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "kv_bytes_per_position.json")))
    fmt = {"f16": mq.F16, "q8_0": mq.Q8_0, "q4_0": mq.Q4_0}
    # 512 K and 512 V elements per position and layer = 4 kv heads x head_dim 128
    pages = 262144 // 32
    for m in g["modes"]:
        k, v = fmt[m["k"]], fmt[m["v"]]
        if (k == mq.F16) != (v == mq.F16):
            continue
        total, planes = mq.kv_cache_bytes(mq.cache_desc(pages, 4, 128, k, v))
        assert total == m["bytes_per_position"] * 262144, m
        assert round(total * g["layers"] / 1e9, 2) == m["session_gb"]
        assert planes[0] + planes[1] == 512 * 262144 * (2 if k == mq.F16 else (34 / 32 if k == mq.Q8_0 else 18 / 32))


def test_cache_bytes_rejects_bad_dimensions():
    assert mq.kv_cache_bytes(mq.cache_desc(0, 8, 128, mq.Q8_0, mq.Q8_0))[0] == 0
    assert mq.kv_cache_bytes(mq.cache_desc(10, 8, 100, mq.Q8_0, mq.Q8_0))[0] == 0
    assert mq.kv_cache_bytes(mq.cache_desc(10, 8, 128, 7, mq.Q8_0))[0] == 0
    d = mq.cache_desc(10, 8, 128, mq.Q8_0, mq.Q8_0)
    d.page_size = 16
    assert mq.kv_cache_bytes(d)[0] == 0


def _fake_cache(num_pages=64, hkv=2, d=128, kf=mq.Q8_0, vf=mq.Q8_0):
    return mq.KVCache(num_pages, hkv, d, kf, vf)


def _desc(c, ok_ptrs=True):
    p = FAKE if ok_ptrs else 0
    return mq.cache_desc(c.num_pages, c.num_kv_heads, c.head_dim, c.k_fmt, c.v_fmt, p, p, p, p)


def _ws(desc, hq, kinds, seqs, offs, max_pages):
    ws = ctypes.c_size_t(0)
    st = mq.load().mixattn_workspace_bytes(ctypes.byref(desc), hq, len(seqs), mq._i32_array(kinds),
                                           mq._i32_array(seqs), mq._i32_array(offs), max_pages,
                                           ctypes.byref(ws))
    return st, ws.value


def test_workspace_sizing_and_row_validation():
    c = _fake_cache()
    d = _desc(c)
    st, ws = _ws(d, 8, [0, 1], [100, 50], [99, 10], 4)
    assert st == mq.OK and ws > 0 and ws % 256 == 0
    # decode row must have q_offset == seq_len - 1
    assert _ws(d, 8, [0], [100], [98], 4)[0] == mq.ERR_INVALID_ARG
    # chunk row needs 0 <= q_offset < seq_len
    assert _ws(d, 8, [1], [100], [100], 4)[0] == mq.ERR_INVALID_ARG
    assert _ws(d, 8, [1], [100], [-1], 4)[0] == mq.ERR_INVALID_ARG
    # unknown row kind, empty batch, too few page-table columns, more pages than the pool
    assert _ws(d, 8, [2], [100], [99], 4)[0] == mq.ERR_INVALID_ARG
    assert _ws(d, 8, [], [], [], 4)[0] == mq.ERR_INVALID_ARG
    assert _ws(d, 8, [0], [129], [128], 4)[0] == mq.ERR_INVALID_ARG
    assert _ws(d, 8, [0], [65 * 32], [65 * 32 - 1], 100)[0] == mq.ERR_INVALID_ARG
    # q heads not a multiple of kv heads; unsupported group size
    assert _ws(d, 7, [0], [100], [99], 4)[0] == mq.ERR_INVALID_ARG
    assert _ws(d, 32, [0], [100], [99], 4)[0] == mq.ERR_UNSUPPORTED
    # zero-length decode row
    assert _ws(d, 8, [0], [0], [-1], 4)[0] == mq.ERR_INVALID_ARG


def test_workspace_grows_with_decode_splits_only():
    c = _fake_cache(num_pages=20000)
    d = _desc(c)
    _, small = _ws(d, 8, [0], [1000], [999], 10000)
    _, big = _ws(d, 8, [0], [300000], [299999], 10000)
    _, chunk = _ws(d, 8, [1], [300000], [299000], 10000)
    assert big > small
    # a chunk row needs no split partials, only its tile descriptors
    assert chunk < big


def test_append_and_run_reject_bad_arguments_without_launching():
    lib = mq.load()
    c = _fake_cache()
    d = _desc(c)
    nul = ctypes.c_void_p(0)
    # n_new == 0 is a no-op that never touches the device
    assert lib.mixattn_kv_append_quant(ctypes.byref(d), nul, nul, nul, 0, nul) == mq.OK
    assert lib.mixattn_kv_append_quant(ctypes.byref(d), nul, nul, nul, -1, nul) == mq.ERR_INVALID_ARG
    p = ctypes.c_void_p(FAKE)
    assert lib.mixattn_kv_append_quant(ctypes.byref(d), nul, p, p, 4, nul) == mq.ERR_INVALID_ARG
    odd = ctypes.c_void_p(FAKE + 2)
    assert lib.mixattn_kv_append_quant(ctypes.byref(d), odd, p, p, 4, nul) == mq.ERR_INVALID_ARG
    bad = _desc(c, ok_ptrs=False)
    assert lib.mixattn_kv_append_quant(ctypes.byref(bad), p, p, p, 4, nul) == mq.ERR_INVALID_ARG
    mis = _desc(c)
    mis.k_quant = FAKE + 16  # plane not 256-byte aligned
    assert lib.mixattn_kv_append_quant(ctypes.byref(mis), p, p, p, 4, nul) == mq.ERR_INVALID_ARG
    f16q = mq.cache_desc(64, 2, 128, mq.F16, mq.Q8_0, FAKE, 0, FAKE, FAKE)
    assert lib.mixattn_kv_append_quant(ctypes.byref(f16q), p, p, p, 4, nul) == mq.ERR_UNSUPPORTED
    assert lib.mixattn_kv_export_blocks(ctypes.byref(d), 2, p, 4, p, nul) == mq.ERR_INVALID_ARG
    assert lib.mixattn_kv_export_blocks(ctypes.byref(d), 0, p, 0, p, nul) == mq.OK
    # plan_create validates rows before touching the device
    h = ctypes.c_void_p(0)
    ws = ctypes.c_size_t(0)
    st = lib.mixattn_plan_create(ctypes.byref(h), ctypes.byref(d), 8, 1, mq._i32_array([0]),
                                 mq._i32_array([100]), mq._i32_array([50]), 4, ctypes.byref(ws))
    assert st == mq.ERR_INVALID_ARG and not h.value
    # run / update / info on a NULL plan
    assert lib.mixattn_run(nul, p, p, p, p, 1 << 20, nul) == mq.ERR_INVALID_ARG
    assert lib.mixattn_plan_info(nul, None, None, None) == mq.ERR_INVALID_ARG
    lib.mixattn_plan_destroy(nul)  # no-op


def test_workload_slots_and_page_table_are_consistent():
    w = wl.tiny()
    pt = wl.page_table(w)
    for r in range(w.n_rows):
        s = wl.slots(w, pt, r, 0, w.seq_lens[r])
        assert len(np.unique(s)) == len(s)
        assert (s // 32 < w.num_pages).all()
