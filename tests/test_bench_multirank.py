"""The bench's multi-GPU host logic on CPU: two gloo ranks (one process per
rank, as a multi-GPU launch runs them) pass the barrier, agree on the
slowest rank's time and report the whole-job rate over it. The sessions are
independent (replicas only), so this is the whole of the cross-rank logic."""
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


def _rank(rank, ws, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=ws)
    try:
        bench.barrier(ws)
        seconds = 1.0 + rank  # rank r took 1 + r seconds for the same 12 frames
        res = {"max": bench.max_over_ranks(seconds, ws), "rate": bench.whole_job_rate(12, seconds, ws)}
        bench.barrier(ws)
    finally:
        dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(res, f)


@pytest.mark.parametrize("ws", [2])
def test_gloo_ranks_agree_on_slowest_time(tmp_path, ws):
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank, args=(r, ws, port, str(tmp_path))) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(ws):
        res = json.load(open(tmp_path / f"rank{r}.json"))
        assert res["max"] == float(ws)  # the slowest rank took ws seconds
        assert res["rate"] == pytest.approx(ws * 12 / ws)  # every rank's frames over the slowest time


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, 1) == 2.5
    assert bench.whole_job_rate(10, 2.0, 1) == 5.0
