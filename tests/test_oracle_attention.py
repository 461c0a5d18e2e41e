"""Pins for the oracle's fp64 attention (CPU only).

The attention the oracle computes is textbook causal softmax attention over the
dequantised cache, with chunk rows and decode rows in one batch (page
"自研RDNA高併發推論引擎 以AI Max+ 395為範例", §1 "統一 mixed-batch 介面").  It is
pinned to torch's fp64 scaled_dot_product_attention (a library routine: causal
mask with a position offset, grouped-query heads), to closed forms, and to the
invariant that a decode row equals the last row of the same sequence run as a
chunk.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl


def _cache_blocks(w, r, fmt_k, fmt_v):
    k, v = wl.row_kv(w, r)
    return oracle.quantize(fmt_k, k), oracle.quantize(fmt_v, v)


def _sdpa_reference(w, kb, vb, window=0):
    """torch fp64 SDPA over the oracle-dequantised K/V, row by row (window > 0:
    a band mask, key j visible to position p iff p - window < j <= p)."""
    q = wl.queries(w)
    out = []
    g = w.num_q_heads // w.num_kv_heads
    for r in range(w.n_rows):
        s, off = w.seq_lens[r], w.q_offsets[r]
        qs = w.q_starts[r]
        qr = torch.from_numpy(q[qs:qs + s - off].astype(np.float64)).permute(1, 0, 2)[None]
        kd = oracle.dequantize(w.k_fmt, kb[r]).reshape(s, w.num_kv_heads, w.head_dim)
        vd = oracle.dequantize(w.v_fmt, vb[r]).reshape(s, w.num_kv_heads, w.head_dim)
        kt = torch.from_numpy(kd).permute(1, 0, 2)[None]
        vt = torch.from_numpy(vd).permute(1, 0, 2)[None]
        pos = torch.arange(off, s)[:, None]
        mask = torch.arange(s)[None, :] <= pos  # key j visible to the query at position p iff j <= p
        if window > 0:
            mask = mask & (torch.arange(s)[None, :] > pos - window)
        o = torch.nn.functional.scaled_dot_product_attention(qr, kt, vt, attn_mask=mask,
                                                             enable_gqa=(g > 1))
        out.append(o[0].permute(1, 0, 2).numpy())
    return np.concatenate(out, axis=0)


@pytest.mark.parametrize("fmt_k,fmt_v", [(wl.FMT_F16, wl.FMT_F16), (wl.FMT_Q8_0, wl.FMT_Q8_0),
                                         (wl.FMT_Q4_0, wl.FMT_Q4_0), (wl.FMT_Q8_0, wl.FMT_Q4_0)])
def test_matches_torch_sdpa_fp64_tiny(fmt_k, fmt_v):
    w = wl.tiny(fmt_k, fmt_v)
    kb, vb = zip(*[_cache_blocks(w, r, fmt_k, fmt_v) for r in range(w.n_rows)])
    got = oracle.attention(fmt_k, fmt_v, wl.queries(w), kb, vb, w.seq_lens, w.q_offsets)
    ref = _sdpa_reference(w, kb, vb)
    assert got.shape == ref.shape == (w.total_q, 4, 64)
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)


def test_matches_torch_sdpa_fp64_gqa8_d128():
    w = wl.custom("g8", 16, 2, 128, wl.FMT_Q8_0, wl.FMT_Q8_0, seed=5,
                  rows=[(wl.ROW_CHUNK, 70, 33), (wl.ROW_DECODE, 45, 44), (wl.ROW_CHUNK, 20, 0)],
                  n_outlier=3)
    kb, vb = zip(*[_cache_blocks(w, r, w.k_fmt, w.v_fmt) for r in range(w.n_rows)])
    got = oracle.attention(w.k_fmt, w.v_fmt, wl.queries(w), kb, vb, w.seq_lens, w.q_offsets)
    np.testing.assert_allclose(got, _sdpa_reference(w, kb, vb), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("fmt", [wl.FMT_F16, wl.FMT_Q8_0, wl.FMT_Q4_0])
def test_single_key_returns_that_value(fmt):
    w = wl.custom("one", 8, 2, 64, fmt, fmt, seed=9, rows=[(wl.ROW_DECODE, 1, 0)])
    kb, vb = _cache_blocks(w, 0, fmt, fmt)
    got = oracle.attention(fmt, fmt, wl.queries(w), [kb], [vb], w.seq_lens, w.q_offsets)
    vd = oracle.dequantize(fmt, vb).reshape(1, 2, 64)
    for h in range(8):
        assert np.array_equal(got[0, h], vd[0, h // 4])


def test_equal_keys_give_the_mean_of_values():
    # all keys identical -> every score equal -> uniform weights over keys 0..p
    w = wl.custom("eq", 4, 1, 64, wl.FMT_Q8_0, wl.FMT_Q8_0, seed=3, rows=[(wl.ROW_CHUNK, 40, 30)])
    k, v = wl.row_kv(w, 0)
    k[:] = k[0]
    kb, vb = oracle.quantize(wl.FMT_Q8_0, k), oracle.quantize(wl.FMT_Q8_0, v)
    got = oracle.attention(wl.FMT_Q8_0, wl.FMT_Q8_0, wl.queries(w), [kb], [vb], w.seq_lens, w.q_offsets)
    vd = oracle.dequantize(wl.FMT_Q8_0, vb).reshape(40, 1, 64)
    for i in range(10):
        p = 30 + i
        np.testing.assert_allclose(got[i], np.repeat(vd[:p + 1, 0].mean(axis=0)[None], 4, axis=0),
                                   rtol=1e-12, atol=1e-14)


def test_decode_row_equals_last_row_of_chunk():
    fmt = wl.FMT_Q4_0
    w_chunk = wl.custom("c", 8, 2, 128, fmt, fmt, seed=21, rows=[(wl.ROW_CHUNK, 97, 50)])
    w_dec = wl.custom("c", 8, 2, 128, fmt, fmt, seed=21, rows=[(wl.ROW_DECODE, 97, 96)])
    kb, vb = _cache_blocks(w_chunk, 0, fmt, fmt)
    kb2, vb2 = _cache_blocks(w_dec, 0, fmt, fmt)
    assert np.array_equal(kb, kb2) and np.array_equal(vb, vb2)
    q = wl.queries(w_chunk)
    oc = oracle.attention(fmt, fmt, q, [kb], [vb], w_chunk.seq_lens, w_chunk.q_offsets)
    od = oracle.attention(fmt, fmt, q[-1:], [kb], [vb], w_dec.seq_lens, w_dec.q_offsets)
    assert np.array_equal(oc[-1], od[0])


def test_identical_queries_in_a_group_give_identical_outputs():
    w = wl.custom("gq", 8, 2, 64, wl.FMT_Q8_0, wl.FMT_Q8_0, seed=4, rows=[(wl.ROW_CHUNK, 33, 0)])
    kb, vb = _cache_blocks(w, 0, w.k_fmt, w.v_fmt)
    q = wl.queries(w)
    q[:, 1] = q[:, 0]
    q[:, 5] = q[:, 6]
    o = oracle.attention(w.k_fmt, w.v_fmt, q, [kb], [vb], w.seq_lens, w.q_offsets)
    assert np.array_equal(o[:, 0], o[:, 1]) and np.array_equal(o[:, 5], o[:, 6])
    # same q in different kv groups sees different keys
    q[:, 4] = q[:, 0]
    o = oracle.attention(w.k_fmt, w.v_fmt, q, [kb], [vb], w.seq_lens, w.q_offsets)
    assert not np.array_equal(o[:, 0], o[:, 4])


def test_selected_rows_match_the_full_evaluation():
    w = wl.tiny()
    kb, vb = zip(*[_cache_blocks(w, r, w.k_fmt, w.v_fmt) for r in range(w.n_rows)])
    q = wl.queries(w)
    full = oracle.attention(w.k_fmt, w.v_fmt, q, kb, vb, w.seq_lens, w.q_offsets)
    sel = np.array([0, 1, 2, 17, 65], dtype=np.int32)
    part = oracle.attention(w.k_fmt, w.v_fmt, q, kb, vb, w.seq_lens, w.q_offsets, sel=sel)
    assert np.array_equal(part, full[sel])


def test_workload_shapes_follow_the_configs():
    w = wl.tiny()
    assert (w.num_q_heads, w.num_kv_heads, w.head_dim) == (4, 1, 64)
    assert w.seq_lens == [100, 300, 192] and w.q_offsets == [99, 299, 128]
    assert w.total_q == 66
    s = wl.serving_mix()
    assert s.n_rows == 17 and s.q_lens[-1] == 2048 and s.q_offsets[-1] == 0
    assert all(1024 <= c <= 32768 for c in s.seq_lens[:16])
    f = wl.fairness()
    assert f.seq_lens[-1] == 202048 and f.q_offsets[-1] == 200000
    assert all(2048 <= c <= 16384 for c in f.seq_lens[:16])
    ls = wl.long_session()
    assert ls.seq_lens[0] == 262144 and all(512 <= c <= 8192 for c in ls.seq_lens[1:])
    pt = wl.page_table(s)
    used = pt[pt >= 0]
    assert len(np.unique(used)) == len(used) == s.num_pages
    # regenerating a token range matches the same range of the full draw
    k, v = wl.row_kv(s, 3)
    k2, v2 = wl.row_kv(s, 3, 4000, 4200)
    assert np.array_equal(k[4000:4200], k2) and np.array_equal(v[4000:4200], v2)


# ---------------------------------------------------------------------------
# Sliding-window attention (the page's per-model table, Gemma 4 row: its SWA
# layers read the same Q8 cache).  Reading: a window of W keys ends at the
# query's own position, keys p - W + 1 .. p.
# ---------------------------------------------------------------------------

def _window_case(fmt_k, fmt_v, seed=13):
    rows = [(wl.ROW_CHUNK, 150, 40), (wl.ROW_DECODE, 300, 299), (wl.ROW_DECODE, 5, 4), (wl.ROW_CHUNK, 70, 0)]
    return wl.custom("win", 8, 2, 64, fmt_k, fmt_v, seed=seed, rows=rows, n_outlier=2)


@pytest.mark.parametrize("window", [1, 2, 31, 32, 33, 100, 1000])
@pytest.mark.parametrize("fmt_k,fmt_v", [(wl.FMT_F16, wl.FMT_F16), (wl.FMT_Q8_0, wl.FMT_Q4_0)])
def test_window_matches_torch_sdpa_band_mask(fmt_k, fmt_v, window):
    w = _window_case(fmt_k, fmt_v)
    kb, vb = zip(*[_cache_blocks(w, r, fmt_k, fmt_v) for r in range(w.n_rows)])
    got = oracle.attention(fmt_k, fmt_v, wl.queries(w), kb, vb, w.seq_lens, w.q_offsets, window=window)
    np.testing.assert_allclose(got, _sdpa_reference(w, kb, vb, window=window), rtol=1e-10, atol=1e-12)


def test_window_of_one_returns_the_own_value():
    fmt = wl.FMT_Q8_0
    w = _window_case(fmt, fmt)
    kb, vb = zip(*[_cache_blocks(w, r, fmt, fmt) for r in range(w.n_rows)])
    got = oracle.attention(fmt, fmt, wl.queries(w), kb, vb, w.seq_lens, w.q_offsets, window=1)
    for r in range(w.n_rows):
        vd = oracle.dequantize(fmt, vb[r]).reshape(w.seq_lens[r], 2, 64)
        for i in range(w.q_lens[r]):
            p = w.q_offsets[r] + i
            for h in range(8):
                assert np.array_equal(got[w.q_starts[r] + i, h], vd[p, h // 4])


def test_window_at_least_the_sequence_is_full_attention():
    fmt = wl.FMT_Q4_0
    w = _window_case(fmt, fmt)
    kb, vb = zip(*[_cache_blocks(w, r, fmt, fmt) for r in range(w.n_rows)])
    q = wl.queries(w)
    full = oracle.attention(fmt, fmt, q, kb, vb, w.seq_lens, w.q_offsets)
    assert np.array_equal(oracle.attention(fmt, fmt, q, kb, vb, w.seq_lens, w.q_offsets, window=300), full)
    assert not np.array_equal(oracle.attention(fmt, fmt, q, kb, vb, w.seq_lens, w.q_offsets, window=299), full)


def test_window_equals_full_attention_over_the_last_keys():
    """A query at position p with window W sees exactly what a decode row sees
    whose cache holds only keys p - W + 1 .. p (the full-attention oracle,
    pinned above, on a truncated cache)."""
    fmt = wl.FMT_Q8_0
    w = _window_case(fmt, fmt)
    kb, vb = zip(*[_cache_blocks(w, r, fmt, fmt) for r in range(w.n_rows)])
    q = wl.queries(w)
    W = 37
    got = oracle.attention(fmt, fmt, q, kb, vb, w.seq_lens, w.q_offsets, window=W)
    for r in (0, 1):
        for i in sorted({0, min(5, w.q_lens[r] - 1), w.q_lens[r] - 1}):
            t = w.q_starts[r] + i
            p = w.q_offsets[r] + i
            lo = max(0, p - W + 1)
            n = p + 1 - lo
            ref = oracle.attention(fmt, fmt, q[t:t + 1], [kb[r][lo:p + 1]], [vb[r][lo:p + 1]], [n], [n - 1])
            assert np.array_equal(got[t], ref[0])
