"""The allocation-free entry point against the workspace entry point.

mixattn_mixed_attention_noalloc serves callers that cannot give the library a
device workspace (a runtime that owns all GPU memory and forbids cudaMalloc, a
serving loop where an allocation would synchronise the device, a plain C host
without a device allocator).  It must give the same outputs as
mixattn_mixed_attention, call after call, although every call reuses the same
library-owned scratch array.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

import workloads as wl
from _harness import TOL, build_cache, oracle_attention

pytestmark = pytest.mark.gpu

D, C = wl.ROW_DECODE, wl.ROW_CHUNK


def _call_noalloc(mq, cache, q, pt_d, w):
    import torch
    o = torch.full_like(q, float("nan"))
    st = mq.load().mixattn_mixed_attention_noalloc(
        ctypes.byref(cache.desc()), w.num_q_heads, ctypes.c_void_p(q.data_ptr()),
        ctypes.c_void_p(pt_d.data_ptr()), int(pt_d.shape[1]), w.n_rows, mq._i32_array(w.seq_lens),
        mq._i32_array(w.q_offsets), mq._i32_array(w.row_kinds), ctypes.c_void_p(o.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == mq.OK, mq.status_string(st)
    torch.cuda.synchronize()
    return o.cpu().numpy()


def test_noalloc_matches_the_workspace_entry_point_on_two_calls_in_a_row():
    import torch
    import mixed_attention_quantized_gb300 as mq
    # several decode rows with many split tiles (so the split counters matter) plus chunk
    # rows, one of them a 5-token verify-style row (verify groups on the workspace path, a
    # tensor-core tile here)
    w = wl.custom("noalloc", 32, 8, 128, wl.FMT_Q8_0, wl.FMT_Q8_0, seed=41,
                  rows=[(D, 9000, 8999), (C, 300, 100), (D, 33, 32), (D, 20000, 19999), (C, 64, 0),
                        (C, 5005, 5000)])
    cache, pt = build_cache(w)
    q = torch.from_numpy(wl.queries(w)).cuda()
    pt_d = torch.from_numpy(pt).cuda()
    ref = mq.mixed_attention(cache, q, pt_d, w.seq_lens, w.q_offsets, w.row_kinds)
    torch.cuda.synchronize()
    ref = ref.cpu().numpy().astype(np.float64)
    mq.device_error(clear=True)
    for _ in range(2):
        got = _call_noalloc(mq, cache, q, pt_d, w)
        assert np.isfinite(got).all()
        assert np.abs(got.astype(np.float64) - ref).max() <= TOL
    assert mq.device_error(clear=True) == 0
    # and against the CPU oracle itself, not only against the other entry point
    assert np.abs(got.astype(np.float64) - oracle_attention(w)).max() <= TOL


def test_noalloc_rejects_a_batch_beyond_its_scratch():
    import torch
    import mixed_attention_quantized_gb300 as mq
    # 256 decode rows at ctx 32768 share one 1024-page cache: 256 x 8 kv heads x 4 split
    # tiles of ~2 KB partials each is ~17 MB of workspace, over the 16 MiB the library
    # holds.  Every input is valid, so the request is refused on its size alone.
    n_rows, ctx = 256, 32768
    cache = mq.KVCache.allocate(ctx // 32, 8, 128, wl.FMT_Q8_0, wl.FMT_Q8_0)
    q = torch.zeros((n_rows, 32, 128), dtype=torch.float16, device="cuda")
    pt = torch.arange(ctx // 32, dtype=torch.int32, device="cuda").repeat(n_rows, 1).contiguous()
    need = mq.workspace_bytes(cache, 32, [D] * n_rows, [ctx] * n_rows, [ctx - 1] * n_rows, ctx // 32)
    assert need > 16 << 20
    with pytest.raises(mq.MixattnError) as e:
        mq.mixed_attention_noalloc(cache, q, pt, [ctx] * n_rows, [ctx - 1] * n_rows, [D] * n_rows)
    assert e.value.status == mq.ERR_WORKSPACE
