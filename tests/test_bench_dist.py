"""The multi-process side of bench.py on CPU: two gloo ranks (world size 2).

bench.py runs one process per GPU under torchrun; the workload is replicated
on every rank (weak scaling) with no collective on the data path.  What ranks
share is the timing: the step time is the slowest rank's and the value is the
units of all ranks over that time.  The reference arm runs on rank 0 only.
These tests run that host logic with the gloo backend; no GPU is needed.
"""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, ws, port):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(ws),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "MKV_DIST_BACKEND": "gloo"})
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)


def _job_value_worker(rank, ws, port, out_dir):
    _env(rank, ws, port)
    import bench
    import torch.distributed as dist
    got_ws, got_rank, _ = bench._dist()
    try:
        ms_local = 10.0 if rank == 0 else 20.0       # rank 1 is the slow one
        ms_step, value = bench._job_value(ms_local, 4, 1000.0, got_ws, "cpu")
        bench._barrier(got_ws)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"ws": got_ws, "rank": got_rank, "ms_step": ms_step, "value": value}, f)
    finally:
        dist.destroy_process_group()


def _reference_worker(rank, ws, port, out_dir):
    _env(rank, ws, port)
    import bench
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--workload", "tiny-4K-b1", "--steps", "1",
                    "--warmup", "3", "--ref-seconds", "0.05"])
    with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
        f.write(buf.getvalue())


def _spawn(fn, tmp_path):
    port = _free_port()
    mp.start_processes(fn, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")


def test_two_ranks_time_is_the_slowest_and_value_sums_ranks(tmp_path):
    _spawn(_job_value_worker, tmp_path)
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    for r, d in enumerate(res):
        assert d["ws"] == 2 and d["rank"] == r
        assert d["ms_step"] == pytest.approx(20.0 / 4)
        # 2 ranks x 1000 units per step over the slowest rank's 5 ms
        assert d["value"] == pytest.approx(2 * 1000.0 / 5e-3)


def test_reference_arm_prints_on_rank_zero_only(tmp_path):
    _spawn(_reference_worker, tmp_path)
    out0 = open(tmp_path / "r0.txt").read().strip().splitlines()
    out1 = open(tmp_path / "r1.txt").read().strip()
    assert out1 == ""
    line = json.loads(out0[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
