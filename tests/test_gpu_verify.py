"""Speculative-verify rows on the GPU against the oracle (reference page
"自研RDNA高併發推論引擎 以AI Max+ 395為範例", §1 "投機解碼（MTP / DFlash）": the
verify pass of a draft runs through the same blocked KV cache).  A verify row
is a short causal chunk -- a handful of draft tokens at an offset.  Up to 24
(query, head) rows it runs on split-K decode-style tiles whose MMA rows are
(query, head) pairs; longer ones keep the 128-row tensor-core tile.  The rows
below cover both.  Bar: max |o - o_oracle| <= 2e-3."""
import numpy as np
import pytest

import workloads as wl
from _harness import TOL, build_cache, max_err, oracle_attention, run_attention

pytestmark = pytest.mark.gpu

D, C = wl.ROW_DECODE, wl.ROW_CHUNK
PAIRS = [(wl.FMT_Q8_0, wl.FMT_Q8_0), (wl.FMT_Q4_0, wl.FMT_Q4_0), (wl.FMT_F16, wl.FMT_F16),
         (wl.FMT_Q8_0, wl.FMT_Q4_0), (wl.FMT_Q4_0, wl.FMT_Q8_0)]


def _verify_rows():
    # 2..16 draft tokens at offsets inside and at the start of a page, contexts from
    # one page to tens of thousands of tokens, mixed with decode rows and a long chunk
    return [(C, 8200, 8184), (C, 30005, 30001), (D, 5000, 4999), (C, 33, 31), (C, 16, 0),
            (C, 12040, 12033), (C, 700, 600), (D, 20, 19)]


@pytest.mark.parametrize("kf,vf", PAIRS)
@pytest.mark.parametrize("hq,hkv", [(32, 8), (16, 2), (8, 8)])
def test_verify_rows_match_oracle(kf, vf, hq, hkv):
    w = wl.custom("verify", hq, hkv, 128, kf, vf, seed=71 + hq + hkv, rows=_verify_rows(), n_outlier=2,
                  spare_pages=5)
    cache, pt = build_cache(w, fill=0xFF)  # stale slots hold NaN patterns
    got = run_attention(w, cache, pt)
    assert max_err(got, oracle_attention(w)) <= TOL


def test_verify_rows_run_on_decode_style_tiles():
    import mixed_attention_quantized_gb300 as mq
    w = wl.custom("verify_tiles", 32, 8, 128, wl.FMT_Q8_0, wl.FMT_Q8_0, 72,
                  [(C, 8200, 8194), (D, 5000, 4999), (C, 40, 36)])
    cache, pt = build_cache(w)
    plan = mq.Plan(cache, 32, w.row_kinds, w.seq_lens, w.q_offsets, pt.shape[1])
    info = plan.info()
    plan.close()
    assert info["chunk_tiles"] == 0 and info["decode_tiles"] > 0
    # a chunk row beyond 24 (query, head) rows keeps the tensor-core tiles
    w2 = wl.custom("verify_tiles2", 32, 8, 128, wl.FMT_Q8_0, wl.FMT_Q8_0, 72, [(C, 8200, 8193)])
    plan = mq.Plan(cache, 32, w2.row_kinds, w2.seq_lens, w2.q_offsets, pt.shape[1])
    assert plan.info()["chunk_tiles"] > 0
    plan.close()


@pytest.mark.parametrize("kf,vf", PAIRS)
def test_last_draft_token_matches_a_decode_row_bit_for_bit(kf, vf):
    """The last query of a verify row and a decode row at the same position run the
    same splits over the same pages; the rows of an MMA and their softmax states are
    independent, so the bits agree."""
    import torch
    wc = wl.custom("v", 32, 8, 128, kf, vf, 73, [(C, 9001, 8995)])
    wd = wl.custom("v", 32, 8, 128, kf, vf, 73, [(D, 9001, 9000)])
    cache, pt = build_cache(wc)
    oc = run_attention(wc, cache, pt)
    qd = torch.from_numpy(wl.row_q(wc, 0)[-1:].copy()).cuda()
    od = run_attention(wd, cache, pt, q=qd)
    assert np.array_equal(oc[-1:], od)
    assert max_err(od, oracle_attention(wc, sel=[5])) <= TOL


def test_verify_row_gives_the_same_bits_alone_and_in_a_batch():
    import torch
    kf = vf = wl.FMT_Q4_0
    rows = [(C, 20000, 19990), (D, 3000, 2999), (C, 800, 792)]
    w = wl.custom("vbatch", 32, 8, 128, kf, vf, 74, rows)
    cache, pt = build_cache(w)
    full = run_attention(w, cache, pt)
    q = wl.queries(w)
    for r in (0, 2):
        sub = wl.custom("one", 32, 8, 128, kf, vf, 74, [rows[r]])
        qr = torch.from_numpy(q[w.q_starts[r]:w.q_starts[r] + w.q_lens[r]].copy()).cuda()
        alone = run_attention(sub, cache, pt[r:r + 1], q=qr)
        assert np.array_equal(alone, full[w.q_starts[r]:w.q_starts[r] + w.q_lens[r]])


@pytest.mark.parametrize("window", [1, 5, 100, 3000])
def test_windowed_verify_rows_match_oracle(window):
    w = wl.custom("vwin", 32, 8, 128, wl.FMT_Q8_0, wl.FMT_Q4_0, 75, _verify_rows())
    cache, pt = build_cache(w)
    got = run_attention(w, cache, pt, window=window)
    assert max_err(got, oracle_attention(w, window=window)) <= TOL
