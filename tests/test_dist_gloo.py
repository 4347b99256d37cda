"""The multi-rank plumbing of bench.py on CPU: two gloo ranks agree on the
slowest rank's time and on the whole-job rate, and the reference arm runs on
rank 0 only.  Batch rows are independent, so the data path has no collective;
these are the only cross-rank steps."""

import json
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2", RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import io
    import contextlib
    import bench
    ws, r, _ = bench.dist_setup()
    ms = [120.0, 150.0][rank]  # rank 1 is the slower one
    bench.barrier(ws)
    m = bench.max_over_ranks(ms, ws, torch.device("cpu"))
    rate = bench.job_rate(m, 100, ws, 384)
    buf = io.StringIO()
    args = type("A", (), {"warmup": 0, "steps": 0, "gpus": 2})()
    with contextlib.redirect_stdout(buf):
        if rank == 1:
            bench.run_reference(args, ws, r)  # must return at once, printing nothing
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"ws": ws, "max": m, "rate": rate, "printed": buf.getvalue()}, f)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.spawn(_worker, args=(port, str(tmp_path)), nprocs=2, join=True)
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    for r in res:
        assert r["ws"] == 2
        assert r["max"] == 150.0
        # 2 ranks x 384 rows per step over 1.5 ms per step
        assert r["rate"] == pytest.approx(2 * 384 / 1.5e-3)
    assert res[1]["printed"] == ""
