"""Sliding-window attention on the GPU against the oracle (reference page
"自研RDNA高併發推論引擎 以AI Max+ 395為範例", §2 per-model table: the Gemma 4
row's SWA layers read the same Q8 cache).  Every query at position p sees keys
p - window + 1 .. p; the planner skips the pages and KV tiles before each
row's window.  Bar: max |o - o_oracle| <= 2e-3, as for full attention."""
import numpy as np
import pytest

import workloads as wl
from _harness import TOL, build_cache, max_err, oracle_attention, run_attention

pytestmark = pytest.mark.gpu

D, C = wl.ROW_DECODE, wl.ROW_CHUNK
PAIRS = [(wl.FMT_Q8_0, wl.FMT_Q8_0), (wl.FMT_Q4_0, wl.FMT_Q4_0), (wl.FMT_F16, wl.FMT_F16),
         (wl.FMT_Q8_0, wl.FMT_Q4_0), (wl.FMT_Q4_0, wl.FMT_Q8_0)]


def _rows():
    # decode rows shorter and longer than the windows, chunk rows whose queries
    # cross a window start, one at offset 0, one long row whose tiles get cut
    return [(D, 1, 0), (D, 33, 32), (D, 1000, 999), (D, 9000, 8999), (C, 300, 100), (C, 70, 0),
            (C, 2500, 2300), (D, 40000, 39999)]


@pytest.mark.parametrize("kf,vf", PAIRS)
@pytest.mark.parametrize("window", [1, 31, 129, 1024, 5000])
def test_windowed_batch_matches_oracle(kf, vf, window):
    w = wl.custom("swa", 32, 8, 128, kf, vf, seed=61 + window, rows=_rows(), n_outlier=2, spare_pages=3)
    cache, pt = build_cache(w, fill=0xFF)  # stale slots hold NaN patterns
    got = run_attention(w, cache, pt, window=window)
    assert max_err(got, oracle_attention(w, window=window)) <= TOL


@pytest.mark.parametrize("window", [64, 100000])
def test_window_beyond_every_row_is_full_attention_bit_for_bit(window):
    """A window at least as long as every row changes nothing, down to the bit
    (64 covers the short rows only: their outputs match the full plan's)."""
    rows = [(D, 50, 49), (C, 60, 20), (D, 64, 63)]
    w = wl.custom("swa_full", 16, 4, 128, wl.FMT_Q8_0, wl.FMT_Q8_0, seed=62, rows=rows)
    cache, pt = build_cache(w)
    assert np.array_equal(run_attention(w, cache, pt, window=window), run_attention(w, cache, pt))


def test_windowed_row_gives_the_same_bits_alone_and_in_a_batch():
    import torch
    kf = vf = wl.FMT_Q4_0
    rows = [(D, 12000, 11999), (C, 900, 500), (D, 77, 76)]
    w = wl.custom("swa_batch", 32, 8, 128, kf, vf, 63, rows)
    cache, pt = build_cache(w)
    full = run_attention(w, cache, pt, window=700)
    q = wl.queries(w)
    for r in (0, 1):
        sub = wl.custom("one", 32, 8, 128, kf, vf, 63, [rows[r]])
        qr = torch.from_numpy(q[w.q_starts[r]:w.q_starts[r] + w.q_lens[r]].copy()).cuda()
        alone = run_attention(sub, cache, pt[r:r + 1], q=qr, window=700)
        assert np.array_equal(alone, full[w.q_starts[r]:w.q_starts[r] + w.q_lens[r]])


def test_windowed_decode_row_matches_last_row_of_the_same_chunk():
    import torch
    kf = vf = wl.FMT_Q8_0
    wc = wl.custom("c", 32, 8, 128, kf, vf, 64, [(C, 5000, 4000)])
    wd = wl.custom("c", 32, 8, 128, kf, vf, 64, [(D, 5000, 4999)])
    cache, pt = build_cache(wc)
    oc = run_attention(wc, cache, pt, window=333)
    qd = torch.from_numpy(wl.row_q(wc, 0)[-1:].copy()).cuda()
    od = run_attention(wd, cache, pt, q=qd, window=333)
    ref = oracle_attention(wc, sel=[999], window=333)
    assert max_err(od, ref) <= TOL and max_err(oc[-1:], ref) <= TOL


def test_window_reads_only_the_pages_it_needs():
    """Pages before a decode row's window are never read: poisoning them (ids
    outside the cache) raises no device error and changes no bit."""
    import mixed_attention_quantized_gb300 as mq
    rows = [(D, 6000, 5999), (C, 400, 300)]
    w = wl.custom("swa_pages", 16, 4, 128, wl.FMT_Q8_0, wl.FMT_Q8_0, 65, rows)
    cache, pt = build_cache(w)
    good = run_attention(w, cache, pt, window=512)
    bad = pt.copy()
    bad[0, :(6000 - 512) // 32] = w.num_pages + 7  # whole pages before the decode row's window
    mq.device_error(clear=True)
    assert np.array_equal(run_attention(w, cache, bad, window=512), good)
    assert mq.device_error(clear=True) == 0
