"""Parity at the measured sizes, in the configuration bench.py times, on outputs
the oracle can compute one by one (every decode row, a spread of chunk rows)."""
import numpy as np
import pytest

import workloads as wl
from _harness import TOL, build_cache, max_err, oracle_attention, run_attention

pytestmark = pytest.mark.gpu


def _chunk_sample(w, n):
    r = w.n_rows - 1
    s0, nq = w.q_starts[r], w.q_lens[r]
    picks = sorted(set([0, 1, 31, 32, 33, 127, 128, nq // 2, nq - 2, nq - 1] +
                       list(np.linspace(0, nq - 1, n).astype(int))))
    return [s0 + i for i in picks if i < nq]


def test_serving_mix_q8():
    w = wl.serving_mix()
    cache, pt = build_cache(w)
    got = run_attention(w, cache, pt)
    sel = list(range(16)) + _chunk_sample(w, 8)
    ref = oracle_attention(w, sel=sel)
    assert max_err(got[sel], ref) <= TOL


@pytest.mark.parametrize("fmt", [wl.FMT_Q8_0, wl.FMT_Q4_0])
def test_long_session(fmt):
    w = wl.long_session(fmt)
    cache, pt = build_cache(w)
    got = run_attention(w, cache, pt)
    ref = oracle_attention(w)  # 16 decode rows, the first at ctx 262144
    assert max_err(got, ref) <= TOL


def test_fairness_q4():
    w = wl.fairness()
    cache, pt = build_cache(w)
    got = run_attention(w, cache, pt)
    sel = list(range(16)) + _chunk_sample(w, 4)
    ref = oracle_attention(w, sel=sel)
    assert max_err(got[sel], ref) <= TOL


@pytest.mark.parametrize("fmt", [wl.FMT_F16, wl.FMT_Q8_0, wl.FMT_Q4_0])
def test_decode_sweep_b4_ctx8192(fmt):
    w = wl.decode_sweep(4, 8192, fmt)
    cache, pt = build_cache(w)
    got = run_attention(w, cache, pt)
    assert max_err(got, oracle_attention(w)) <= TOL


@pytest.mark.parametrize("fmt", [wl.FMT_F16, wl.FMT_Q8_0, wl.FMT_Q4_0])
def test_decode_sweep_b64_ctx65536_sampled(fmt):
    """The largest decode-sweep point (64 rows x 65536 tokens; 17 GB of fp16 KV at the
    fp16 end) in the bench's launch configuration; the oracle evaluates a spread of
    rows one by one."""
    w = wl.decode_sweep(64, 65536, fmt)
    cache, pt = build_cache(w, append_tokens=65536)
    got = run_attention(w, cache, pt)
    sel = [0, 1, 17, 31, 32, 50, 62, 63]
    assert max_err(got[sel], oracle_attention(w, sel=sel)) <= TOL


@pytest.mark.parametrize("kf,vf", [(wl.FMT_Q8_0, wl.FMT_Q4_0), (wl.FMT_Q4_0, wl.FMT_Q8_0)])
def test_serving_mix_mixed_formats(kf, vf):
    """The serving mix with K8V4 and K4V8 caches: every decode row and a spread of
    chunk rows against the oracle."""
    w = wl.serving_mix(kf, vf)
    cache, pt = build_cache(w)
    got = run_attention(w, cache, pt)
    sel = list(range(16)) + _chunk_sample(w, 8)
    assert max_err(got[sel], oracle_attention(w, sel=sel)) <= TOL
