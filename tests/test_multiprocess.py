"""The N > 1 path of bench.py on CPU: world size 2 over gloo.

Each rank runs its own batch (replicas; the attention step has no exchange
between sequences), so the only cross-rank operations are the barrier and the
max-over-ranks of the step time; rank 0 alone prints the JSON line.
"""
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import io
    import contextlib
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = 10.0 + 5.0 * rank  # the slower rank sets the job's time
    dist.barrier()
    ms = bench.max_over_ranks(local_ms)
    value = bench.whole_job_tokens_per_s(2064, world, ms)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.emit({"value": value, "ms_per_step": ms, "n_gpus": world}, rank)
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(buf.getvalue())
    dist.barrier()
    dist.destroy_process_group()


def test_world_size_two_gloo(tmp_path):
    port = _free_port()
    mp.spawn(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    out0 = (tmp_path / "rank0.txt").read_text().strip().splitlines()
    out1 = (tmp_path / "rank1.txt").read_text().strip()
    assert out1 == ""
    assert len(out0) == 1
    line = json.loads(out0[0])
    assert line["ms_per_step"] == 15.0
    assert line["n_gpus"] == 2
    assert abs(line["value"] - 2 * 2064 / 0.015) < 1e-6


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_tokens_per_s(16, 1, 2.0) == 8000.0
