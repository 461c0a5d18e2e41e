"""The fair batch builder (include/mixattn_sched.h) on the CPU, one test per
rule of the reference page "自研RDNA高併發推論引擎 以AI Max+ 395為範例" (§1
"公平性：排隊不插隊" and the "排程器保證什麼" table), plus a fake-clock run of
the page's fairness scenario (a short request behind a 250k-token prompt) and
a check that every batch it builds is accepted by the attention ABI's own
validation.  No GPU is used."""
import numpy as np
import pytest

import mixed_attention_quantized_gb300 as mq

D, C = mq.ROW_DECODE, mq.ROW_CHUNK


def run_until(b, pred, limit=100000):
    """Step the builder until pred(batch) holds; returns (batch, steps taken)."""
    for i in range(limit):
        bt = b.next_batch()
        if pred(bt):
            return bt, i
        if bt.kind != mq.STEP_IDLE:
            b.complete()
    raise AssertionError("condition never reached")


def drain(b, limit=100000):
    """Run to idle; returns the list of batches."""
    out = []
    for _ in range(limit):
        bt = b.next_batch()
        if bt.kind == mq.STEP_IDLE:
            return out
        out.append(bt)
        b.complete()
    raise AssertionError("builder never went idle")


def test_default_config_is_the_pages():
    c = mq.FairBatchBuilder.default_config()
    assert (c.prefill_chunk, c.near_done_tokens, c.max_pending_per_client, c.max_decode_rows) == (512, 64, 0, 0)


def test_rows_follow_the_attention_abi_positions():
    b = mq.FairBatchBuilder(max_sessions=2, prefill_chunk=4)
    b.submit(1, 0, 10, 3)
    batches = drain(b)
    # prompt slices 0-4, 4-8, 8-10, then decode rows at positions 10 and 11
    rows = [(k, s, o) for bt in batches for k, s, o in zip(bt.row_kinds, bt.seq_lens, bt.q_offsets)]
    assert rows == [(C, 4, 0), (C, 8, 4), (C, 10, 8), (D, 11, 10), (D, 12, 11)]
    info = b.info(1)
    assert info["state"] == mq.REQ_DONE and info["generated"] == 3 and info["cached"] == 12
    assert info["first_token_step"] == 2 and info["done_step"] == 4


def test_bounded_chunk_feeds_a_long_prompt_one_slice_per_step():
    b = mq.FairBatchBuilder(max_sessions=4, prefill_chunk=512)
    b.submit(1, 0, 250000, 1)
    batches = drain(b)
    chunks = [(s, o) for bt in batches for k, s, o in zip(bt.row_kinds, bt.seq_lens, bt.q_offsets) if k == C]
    assert len(chunks) == -(-250000 // 512)
    assert all(sum(k == C for k in bt.row_kinds) <= 1 for bt in batches)
    assert all(s - o <= 512 for s, o in chunks)
    assert [o for _, o in chunks] == [0] + [s for s, _ in chunks[:-1]]  # contiguous slices
    assert chunks[-1][0] == 250000


def test_decode_first_no_due_decoder_waits_behind_a_chunk():
    """With a cap of 2 decode rows and 4 due decoders, the step carries no chunk;
    the chunk joins the step that serves the last due decoders."""
    b = mq.FairBatchBuilder(max_sessions=5, prefill_chunk=8, max_decode_rows=2)
    for i in range(4):
        b.submit(i, i, 4, 1000)  # short prompts: decoders after one slice each
    while b.counts()["decoders"] < 4:
        assert b.next_batch().kind != mq.STEP_IDLE
        b.complete()
    # the step that made the fourth decoder carried a chunk: all four are due
    b.submit(99, 9, 4000, 10)
    bt = b.next_batch()
    assert bt.kind == mq.STEP_DECODE and bt.row_kinds == [D, D]
    first = set(bt.request_ids)
    b.complete()
    bt = b.next_batch()
    assert bt.kind == mq.STEP_MERGED and bt.row_kinds == [D, D, C] and bt.request_ids[-1] == 99
    assert first | set(bt.request_ids[:2]) == {0, 1, 2, 3}
    b.complete()


def test_decode_first_invariant_over_a_random_trace():
    """Property over a seeded random workload: a step with a chunk never leaves a
    due decoder unserved (the row set of a merged step holds every decoder that
    was due), and decode rows never exceed the cap."""
    rng = np.random.default_rng(7)
    b = mq.FairBatchBuilder(max_sessions=6, prefill_chunk=64, max_decode_rows=3)
    nid = 0
    due = set()  # mirror of the due flags: set after a chunk step, cleared when served
    decoders = set()
    for step in range(3000):
        if rng.random() < 0.05:
            b.submit(nid, int(rng.integers(0, 3)), int(rng.integers(1, 600)), int(rng.integers(1, 200)))
            nid += 1
        bt = b.next_batch()
        if bt.kind == mq.STEP_IDLE:
            continue
        served = {i for i, k in zip(bt.request_ids, bt.row_kinds) if k == D}
        assert len(served) <= 3
        if C in bt.row_kinds:
            assert due <= served, (step, due - served)
        due -= served
        b.complete()
        decoders = {i for i in range(nid) if b.info(i)["state"] == mq.REQ_DECODE}
        if C in bt.row_kinds:
            due = set(decoders)
        else:
            due &= decoders
        # fresh decoders (prompt completed this step) are due too
        due |= {i for i in decoders if b.info(i)["first_token_step"] == b.counts()["steps"] - 1}


def test_srtf_near_done_prefill_goes_first_fifo_within_class():
    b = mq.FairBatchBuilder(max_sessions=4, prefill_chunk=100)
    b.submit(1, 0, 5000, 1)  # long, admitted first
    b.submit(2, 1, 80, 1)    # near-done (<= one chunk)
    b.submit(3, 2, 60, 1)    # near-done, admitted after 2
    order = [bt.request_ids[-1] for bt in drain(b) if C in bt.row_kinds]
    assert order[:2] == [2, 3]  # near-done class first, FIFO within it
    assert order[2] == 1
    # a long prefill whose remainder falls to one chunk becomes near-done
    b2 = mq.FairBatchBuilder(max_sessions=4, prefill_chunk=100)
    b2.submit(1, 0, 250, 1)
    b2.submit(2, 1, 300, 1)
    order = [bt.request_ids[-1] for bt in drain(b2) if C in bt.row_kinds]
    assert order == [1, 1, 1, 2, 2, 2]  # long FIFO; then request 1 (50 left) is near-done


def test_starvation_preemption_behind_the_near_done_gate():
    def setup(limit_short):
        b = mq.FairBatchBuilder(max_sessions=2, prefill_chunk=64, near_done_tokens=64)
        b.submit(1, 0, 10, limit_short)  # becomes a decoder quickly
        b.submit(2, 1, 100000, 1)        # a long prompt, resident
        run_until(b, lambda bt: b.info(1)["state"] == mq.REQ_DECODE)
        b.complete()
        b.submit(3, 2, 10, 1)            # waits for a slot: both slots are taken
        return b

    # a resident decoder within 64 tokens of its limit: long slices yield
    b = setup(limit_short=50)
    assert b.counts()["waiting"] == 1
    bt = b.next_batch()
    assert C not in bt.row_kinds and bt.request_ids == [1]
    b.complete()
    run_until(b, lambda bt: b.info(3)["state"] != mq.REQ_WAITING)  # the decoder finished, 3 admitted
    assert b.info(2)["cached"] == 64  # the long prompt did not advance while preempted (one slice before)

    # only long-output decoders resident: no preemption, the long prompt advances
    b = setup(limit_short=10000)
    bt = b.next_batch()
    assert C in bt.row_kinds and bt.request_ids[-1] == 2


def test_mark_all_decoders_due_after_a_step_with_a_chunk():
    b = mq.FairBatchBuilder(max_sessions=5, prefill_chunk=16, max_decode_rows=0)
    for i in range(3):
        b.submit(i, i, 8, 1000)
    run_until(b, lambda bt: b.counts()["decoders"] == 3)  # a decode step serving all three
    b.complete()
    b.submit(10, 5, 10000, 5)
    # every decoder was served in this rotation: the first slice runs alone, then all are due again
    bt = b.next_batch()
    assert bt.kind == mq.STEP_PREFILL and bt.request_ids == [10]
    b.complete()
    for _ in range(20):
        bt = b.next_batch()
        assert set(bt.request_ids[:3]) == {0, 1, 2} and bt.row_kinds[:3] == [D, D, D]
        assert bt.kind == mq.STEP_MERGED  # every decoder fits: each step also carries a slice
        b.complete()


def test_pop_decoder_rotation_serves_everyone_equally():
    b = mq.FairBatchBuilder(max_sessions=5, prefill_chunk=16, max_decode_rows=2)
    for i in range(4):
        b.submit(i, i, 8, 100000)
    run_until(b, lambda bt: b.counts()["decoders"] == 4)
    b.complete()
    served = {i: 0 for i in range(4)}
    steps_ids = []
    for _ in range(40):
        bt = b.next_batch()
        steps_ids.append(bt.request_ids)
        for i in bt.request_ids:
            served[i] += 1
        b.complete()
    assert max(served.values()) - min(served.values()) <= 1
    # no decoder is served twice while another waits: two consecutive steps serve all four
    assert all(set(a) | set(c) == {0, 1, 2, 3} for a, c in zip(steps_ids, steps_ids[1:]))


def test_client_quota_and_cross_client_admission():
    b = mq.FairBatchBuilder(max_sessions=1, prefill_chunk=1000, max_pending_per_client=2)
    assert b.submit(1, 7, 10, 1) == mq.OK
    assert b.submit(2, 7, 10, 1) == mq.OK
    assert b.submit(3, 7, 10, 1) == mq.ERR_CLIENT_QUOTA  # the page's client_quota
    assert b.submit(4, 8, 10, 1) == mq.OK
    assert b.submit(5, 8, 10, 1) == mq.OK
    with pytest.raises(mq.MixattnError):
        b.info(3)  # refused requests are not queued
    order = [bt.request_ids[0] for bt in drain(b)]
    assert order == [1, 4, 2, 5]  # one slot: admission alternates between the clients


def test_invalid_arguments_are_rejected():
    with pytest.raises(mq.MixattnError):
        mq.FairBatchBuilder(max_sessions=0)
    b = mq.FairBatchBuilder(max_sessions=2)
    assert b.submit(1, 0, 10, 1) == mq.OK
    with pytest.raises(mq.MixattnError):
        b.submit(1, 0, 10, 1)  # duplicate id
    with pytest.raises(mq.MixattnError):
        b.submit(2, 0, 0, 1)
    with pytest.raises(mq.MixattnError):
        b.complete()  # nothing built
    b.next_batch()
    with pytest.raises(mq.MixattnError):
        b.next_batch()  # the built step was not completed


def fake_clock_ttft(long_prompt, chunk=512, near_done=64):
    """The page's five-into-four fairness scenario under a fake clock: a long
    prompt arrives first, then four short requests, with four session slots, so
    the fourth short request waits for a slot.  A step costs 2 ms + 0.02 ms per
    token it processes.  Returns the short requests' TTFT in ms."""
    b = mq.FairBatchBuilder(max_sessions=4, prefill_chunk=chunk, near_done_tokens=near_done)
    t = 0.0
    b.submit(0, 0, long_prompt, 200)
    arrive = {}
    for i in range(1, 5):
        b.submit(i, i, 300, 40)
        arrive[i] = t
    ttft = {}
    while len(ttft) < 4:
        bt = b.next_batch()
        assert bt.kind != mq.STEP_IDLE
        t += 2.0 + 0.02 * sum(s - o for s, o in zip(bt.seq_lens, bt.q_offsets))
        b.complete()
        for i in range(1, 5):
            if i not in ttft and b.info(i)["generated"] >= 1:
                ttft[i] = t - arrive[i]
    return ttft


def test_short_request_ttft_does_not_grow_with_a_long_prompt_ahead():
    """With bounded slices and SRTF the short requests' first tokens do not wait
    for the long prompt, whatever its length; fed whole (one unbounded slice),
    their wait grows with it.  The near-done gate lets the waiting request in
    sooner: resident short decoders (40-token limit, inside the 64-token gate)
    drain without long slices in their steps."""
    fair_50k = fake_clock_ttft(50000)
    fair_250k = fake_clock_ttft(250000)
    assert fair_250k == pytest.approx(fair_50k)
    unbounded = fake_clock_ttft(250000, chunk=1 << 30)
    assert min(unbounded.values()) > 10 * max(fair_250k.values())
    no_gate = fake_clock_ttft(250000, near_done=0)
    assert fair_250k[4] < 0.5 * no_gate[4]  # the request that waited for a slot
    assert [fair_250k[i] for i in (1, 2, 3)] == pytest.approx([no_gate[i] for i in (1, 2, 3)])


def test_every_built_batch_passes_the_attention_abi_validation():
    """The row arrays go straight into the planner: the host-side sizing call of
    the attention ABI accepts every batch of a random trace."""
    rng = np.random.default_rng(3)
    b = mq.FairBatchBuilder(max_sessions=8, prefill_chunk=256, max_decode_rows=6)
    for i in range(24):
        b.submit(i, i % 5, int(rng.integers(1, 3000)), int(rng.integers(1, 80)))
    n = 0
    for bt in drain(b):
        max_pages = max(-(-s // 32) for s in bt.seq_lens)
        ws = mq.workspace_bytes(mq.KVCache(1 << 16, 8, 128, mq.Q8_0, mq.Q8_0), 32, bt.row_kinds, bt.seq_lens,
                                bt.q_offsets, max_pages)
        assert ws > 0
        n += 1
    assert n > 50
