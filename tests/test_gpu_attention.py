"""Parity of the mixed-batch attention step (CUDA, through the C ABI) with the
fp64 oracle over the oracle-dequantised cache, plus the invariants the
reference page relies on (page "自研RDNA高併發推論引擎 以AI Max+ 395為範例":
§1 mixed batch and bit-identical greedy output under concurrency; §2 blocked
KV formats).  Bar: max |o_gpu - o_oracle| <= 2e-3 on fp16 outputs."""
import numpy as np
import pytest

import workloads as wl
from _harness import TOL, build_cache, max_err, oracle_attention, run_attention

pytestmark = pytest.mark.gpu

PAIRS = [(wl.FMT_Q8_0, wl.FMT_Q8_0), (wl.FMT_Q4_0, wl.FMT_Q4_0), (wl.FMT_F16, wl.FMT_F16),
         (wl.FMT_Q8_0, wl.FMT_Q4_0), (wl.FMT_Q4_0, wl.FMT_Q8_0)]
D, C = wl.ROW_DECODE, wl.ROW_CHUNK


@pytest.mark.parametrize("kf,vf", PAIRS)
def test_tiny_config_matches_oracle(kf, vf):
    w = wl.tiny(kf, vf)
    cache, pt = build_cache(w)
    got = run_attention(w, cache, pt)
    ref = oracle_attention(w)
    assert max_err(got, ref) <= TOL


def _ragged(kf, vf, hq, hkv, d, seed):
    rows = [(D, 1, 0), (D, 31, 30), (D, 32, 31), (D, 33, 32), (C, 100, 37), (D, 1000, 999),
            (C, 45, 0), (C, 500, 200), (D, 4097, 4096), (C, 1, 0), (C, 129, 127)]
    return wl.custom(f"ragged_g{hq // hkv}_d{d}", hq, hkv, d, kf, vf, seed, rows, n_outlier=2,
                     spare_pages=7)


@pytest.mark.parametrize("kf,vf", PAIRS)
@pytest.mark.parametrize("hq,hkv,d", [(16, 4, 128), (8, 8, 64), (16, 8, 128), (16, 2, 64)])
def test_ragged_batches_match_oracle(kf, vf, hq, hkv, d):
    w = _ragged(kf, vf, hq, hkv, d, seed=hq * 100 + hkv * 10 + d + kf * 3 + vf)
    cache, pt = build_cache(w, fill=0xFF)  # stale slots hold NaN patterns
    got = run_attention(w, cache, pt)
    ref = oracle_attention(w)
    assert max_err(got, ref) <= TOL


def test_stale_slots_do_not_change_a_bit():
    for kf, vf in PAIRS:
        w = _ragged(kf, vf, 16, 4, 128, seed=77)
        c0, pt = build_cache(w, fill=0)
        c1, _ = build_cache(w, fill=0xFF)
        assert np.array_equal(run_attention(w, c0, pt), run_attention(w, c1, pt))


def test_page_placement_does_not_change_a_bit():
    w = _ragged(wl.FMT_Q8_0, wl.FMT_Q8_0, 16, 4, 128, seed=5)
    c0, pt0 = build_cache(w)
    perm = np.random.default_rng(99).permutation(w.num_pages).astype(np.int32)
    pt1 = np.where(pt0 >= 0, perm[np.maximum(pt0, 0)], -1).astype(np.int32)
    c1, _ = build_cache(w, pt=pt1)
    assert np.array_equal(run_attention(w, c0, pt0), run_attention(w, c1, pt1))


def test_a_row_gives_the_same_bits_alone_and_in_a_batch():
    """The page's greedy outputs stay bit-identical when a request runs alone or
    concurrently; here: a row's output does not depend on the rest of the batch."""
    kf = vf = wl.FMT_Q4_0
    rows = [(D, 5000, 4999), (C, 700, 300), (D, 77, 76), (C, 64, 0), (D, 40000, 39999)]
    w = wl.custom("batch", 32, 8, 128, kf, vf, 11, rows)
    import torch
    cache, pt = build_cache(w)
    full = run_attention(w, cache, pt)
    q = wl.queries(w)
    starts = w.q_starts
    for r in (0, 1, 4):
        sub = wl.custom("one", 32, 8, 128, kf, vf, 11, [rows[r]])
        qr = torch.from_numpy(q[starts[r]:starts[r] + w.q_lens[r]].copy()).cuda()
        alone = run_attention(sub, cache, pt[r:r + 1], q=qr)
        assert np.array_equal(alone, full[starts[r]:starts[r] + w.q_lens[r]])


def test_decode_row_matches_last_row_of_the_same_chunk():
    kf = vf = wl.FMT_Q8_0
    wc = wl.custom("c", 32, 8, 128, kf, vf, 21, [(C, 3000, 2000)])
    wd = wl.custom("c", 32, 8, 128, kf, vf, 21, [(D, 3000, 2999)])
    cache, pt = build_cache(wc)
    oc = run_attention(wc, cache, pt)
    from workloads import row_q
    import torch
    qd = torch.from_numpy(row_q(wc, 0)[-1:].copy()).cuda()
    od = run_attention(wd, cache, pt, q=qd)
    assert np.abs(oc[-1].astype(np.float64) - od[0].astype(np.float64)).max() <= TOL
    ref = oracle_attention(wc, sel=[999])
    assert max_err(od, ref) <= TOL and max_err(oc[-1:], ref) <= TOL


def test_bad_page_id_sets_the_device_error():
    import torch
    import mixed_attention_quantized_gb300 as mq
    w = wl.custom("bad", 8, 2, 64, wl.FMT_Q8_0, wl.FMT_Q8_0, 3, [(D, 100, 99), (C, 80, 40)])
    cache, pt = build_cache(w)
    mq.device_error(clear=True)
    bad = pt.copy()
    bad[0, 1] = w.num_pages + 5
    bad[1, 0] = -3
    out = run_attention(w, cache, bad)
    # the good pages still produced numbers of the right shape
    assert out.shape == (w.total_q, 8, 64)
    # the next call sees that a device check fired and launches nothing
    with pytest.raises(mq.MixattnError) as e:
        run_attention(w, cache, pt)
    assert e.value.status == mq.ERR_DEVICE_CHECK
    with pytest.raises(mq.MixattnError) as e:
        k, v = wl.row_kv(w, 0, 0, 1)
        mq.kv_append_quant(cache, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                           torch.zeros(1, dtype=torch.int32, device="cuda"))
    assert e.value.status == mq.ERR_DEVICE_CHECK
    assert mq.device_error(clear=True) & mq.DEVERR_PAGE_ID
    assert mq.device_error(clear=True) == 0
    # cleared: calls run again
    assert max_err(run_attention(w, cache, pt), oracle_attention(w)) <= TOL


def test_one_call_entry_point_matches_the_plan_path():
    import torch
    import mixed_attention_quantized_gb300 as mq
    w = _ragged(wl.FMT_Q8_0, wl.FMT_Q4_0, 16, 4, 128, seed=1)
    cache, pt = build_cache(w)
    q = torch.from_numpy(wl.queries(w)).cuda()
    o = mq.mixed_attention(cache, q, torch.from_numpy(pt).cuda(), w.seq_lens, w.q_offsets, w.row_kinds)
    torch.cuda.synchronize()
    assert np.array_equal(o.cpu().numpy(), run_attention(w, cache, pt))


def test_plan_update_and_reuse_across_layers():
    import torch
    import mixed_attention_quantized_gb300 as mq
    w1 = _ragged(wl.FMT_Q8_0, wl.FMT_Q8_0, 16, 4, 128, seed=2)
    cache, pt = build_cache(w1)
    ref1 = run_attention(w1, cache, pt)
    plan = mq.Plan(cache, 16, w1.row_kinds, w1.seq_lens, w1.q_offsets, pt.shape[1])
    ws = mq.alloc_workspace(plan.workspace_bytes)
    q = torch.from_numpy(wl.queries(w1)).cuda()
    ptd = torch.from_numpy(pt).cuda()
    outs = []
    for _ in range(3):  # same plan, three "layers"
        o = torch.empty_like(q)
        plan.run(q, ptd, o, ws)
        outs.append(o)
    torch.cuda.synchronize()
    for o in outs:
        assert np.array_equal(o.cpu().numpy(), ref1)
    # re-tile for a smaller batch (first two rows)
    plan.update(w1.row_kinds[:2], w1.seq_lens[:2], w1.q_offsets[:2], pt.shape[1])
    o2 = torch.empty_like(q[:2])
    plan.run(q[:2], ptd[:2], o2, mq.alloc_workspace(plan.workspace_bytes))
    torch.cuda.synchronize()
    assert np.array_equal(o2.cpu().numpy(), ref1[:2])
    plan.close()


def test_workspace_too_small_is_rejected():
    import torch
    import mixed_attention_quantized_gb300 as mq
    w = wl.tiny()
    cache, pt = build_cache(w)
    plan = mq.Plan(cache, 4, w.row_kinds, w.seq_lens, w.q_offsets, pt.shape[1])
    q = torch.from_numpy(wl.queries(w)).cuda()
    with pytest.raises(mq.MixattnError) as e:
        plan.run(q, torch.from_numpy(pt).cuda(), torch.empty_like(q), mq.alloc_workspace(plan.workspace_bytes - 256))
    assert e.value.status == mq.ERR_WORKSPACE


def test_cut_chunk_tiles_match_oracle_and_stay_row_independent():
    """A long chunk row with fewer tiles than SMs has the key range of each tile
    cut into pieces whose partial results merge by log-sum-exp; the result still
    matches the oracle, and the cut depends on the row alone, so the row's bits
    are the same alone and in a batch."""
    import torch
    import mixed_attention_quantized_gb300 as mq
    kf = vf = wl.FMT_Q8_0
    rows = [(C, 8192 + 256, 8192), (D, 5000, 4999)]
    w = wl.custom("cut", 32, 8, 128, kf, vf, 31, rows)
    cache, pt = build_cache(w)
    plan = mq.Plan(cache, 32, w.row_kinds, w.seq_lens, w.q_offsets, pt.shape[1])
    assert plan.info()["chunk_tiles"] > 64  # 64 tiles (256 tokens x 8 kv heads / 32), cut
    plan.close()
    full = run_attention(w, cache, pt)
    assert max_err(full, oracle_attention(w)) <= TOL
    one = wl.custom("cut1", 32, 8, 128, kf, vf, 31, rows[:1])
    q = torch.from_numpy(wl.queries(w)[:256].copy()).cuda()
    alone = run_attention(one, cache, pt[:1], q=q)
    assert np.array_equal(alone, full[:256])


@pytest.mark.parametrize("kf,vf", [(wl.FMT_Q8_0, wl.FMT_Q8_0), (wl.FMT_Q4_0, wl.FMT_Q4_0), (wl.FMT_Q8_0, wl.FMT_Q4_0)])
def test_values_near_the_fp16_limit_stay_finite(kf, vf):
    """V values up to 6e4 (block scales near the largest a format can hold) and
    queries x4 (sharp scores, frequent new maxima): weights relative to a lagging
    softmax reference times those scales must stay inside fp16, and the error
    scales with the values (the 2e-3 budget per unit of V, plus the fp16 rounding
    of the output itself)."""
    gain = 12000.0
    rows = [(D, 3000, 2999), (D, 700, 699), (D, 33, 32), (C, 300, 200)]
    w = wl.custom("near_limit", 32, 8, 128, kf, vf, 21, rows, v_gain=gain, q_gain=4.0)
    cache, pt = build_cache(w)
    out = run_attention(w, cache, pt).astype(np.float64)
    ref = oracle_attention(w)
    assert np.isfinite(out).all()
    assert (np.abs(out - ref) <= TOL * gain + np.abs(ref) * 2.0 ** -11).all(), np.abs(out - ref).max()



LIMIT_PAIRS = [(wl.FMT_Q8_0, wl.FMT_Q8_0), (wl.FMT_Q8_0, wl.FMT_Q4_0), (wl.FMT_Q4_0, wl.FMT_Q8_0),
               (wl.FMT_Q4_0, wl.FMT_Q4_0)]
LIMIT_GAIN = 30000.0  # ~3% of the values clip at +-65504: most blocks hold the largest fp16 value


def _limit_workload(kf, vf, which, rows, seed=23):
    # K at the limit: queries scaled by 1e-4 keep the scores O(1) (K x 3e4 x Q x 1e-4),
    # so the fp32 accumulation of scores stays far inside the budget; unscaled, scores of
    # ~1e4 carry fp32 rounding of ~1e-3 each, which the softmax turns into output errors
    # of ~1e-2 on any fp32-accumulating implementation
    gains = {"k_gain": LIMIT_GAIN, "q_gain": 1e-4} if which == "k" else {"v_gain": LIMIT_GAIN}
    return wl.custom(f"limit_{which}", 32, 8, 128, kf, vf, seed, rows, **gains)


def _limit_bound(which, ref):
    """Errors scale with the values: the 2e-3 budget per unit of V (V at the limit),
    plus the fp16 rounding of the output itself (saturating at 65504)."""
    return TOL * (LIMIT_GAIN if which == "v" else 1.0) + np.abs(ref) * 2.0 ** -11


@pytest.mark.parametrize("kf,vf", LIMIT_PAIRS)
@pytest.mark.parametrize("which", ["k", "v"])
def test_blocks_holding_the_largest_fp16_value_match_oracle(kf, vf, which):
    """K or V blocks whose largest element is +-65504: a Q8_0 scale of 516 and a
    dequantised 127 * 516 = 65532, beyond the fp16 range, in decode rows and in
    chunk rows (the chunk path splits every value into fp16 halves, whose high
    half must not overflow).  Every output is finite and within the oracle's
    value-scaled bound."""
    rows = [(D, 3000, 2999), (D, 700, 699), (D, 33, 32), (C, 300, 200), (C, 129, 0)]
    w = _limit_workload(kf, vf, which, rows)
    k, v = wl.row_kv(w, 0)
    x = (k if which == "k" else v).astype(np.float32)
    assert (np.abs(x) == wl.FP16_MAX).any()  # the inputs do reach the limit
    cache, pt = build_cache(w)
    out = run_attention(w, cache, pt).astype(np.float64)
    ref = oracle_attention(w)
    assert np.isfinite(out).all()
    err = np.abs(out - ref)
    assert (err <= _limit_bound(which, ref)).all(), err.max()


@pytest.mark.parametrize("kf,vf", [(wl.FMT_Q8_0, wl.FMT_Q8_0), (wl.FMT_Q8_0, wl.FMT_Q4_0), (wl.FMT_Q4_0, wl.FMT_Q8_0)])
@pytest.mark.parametrize("which", ["k", "v"])
def test_decode_row_matches_last_chunk_row_at_the_fp16_limit(kf, vf, which):
    """The invariant a decode row == the last row of the same sequence run as a
    chunk, on blocks holding +-65504 (decode tiles keep scales in fp32; chunk
    tiles use the fp16 hi/lo split)."""
    import torch
    wc = _limit_workload(kf, vf, which, [(C, 3000, 2000)], seed=29)
    wd = _limit_workload(kf, vf, which, [(D, 3000, 2999)], seed=29)
    cache, pt = build_cache(wc)
    oc = run_attention(wc, cache, pt).astype(np.float64)
    qd = torch.from_numpy(wl.row_q(wc, 0)[-1:].copy()).cuda()
    od = run_attention(wd, cache, pt, q=qd).astype(np.float64)
    assert np.isfinite(oc).all() and np.isfinite(od).all()
    ref = oracle_attention(wc, sel=[999])
    bound = _limit_bound(which, ref)
    assert (np.abs(od - ref) <= bound).all() and (np.abs(oc[-1:] - ref) <= bound).all()
    assert (np.abs(oc[-1:] - od) <= 2 * bound).all()
