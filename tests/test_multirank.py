"""The bench's N > 1 host logic on CPU: world_size-2 process groups over gloo
(127.0.0.1), no GPU.  Replicas: each rank draws its own inputs, the timing
is the maximum over ranks, the job's value counts every rank's tokens, and
the reference arm runs on rank 0 alone."""
import contextlib
import io
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _worker(rank, ws, port, q):
    try:
        sys.path.insert(0, ROOT)
        os.environ.update(RANK=str(rank), WORLD_SIZE=str(ws), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                          MASTER_PORT=str(port))
        import bench
        got_ws, got_rank, got_local = bench.dist_env()
        assert (got_ws, got_rank, got_local) == (ws, rank, rank)
        dist.init_process_group("gloo", rank=rank, world_size=ws)
        # the slowest rank's time is the job's time
        my_ms = 10.0 + 5.0 * rank
        t_max = bench._max_over_ranks(torch, torch.device("cpu"), ws, my_ms)
        # replicas draw their own inputs
        seed, offsets = bench.replica_inputs(rank, 2000, 8)
        mine = torch.tensor([seed] + offsets, dtype=torch.int64)
        all_inputs = [torch.empty_like(mine) for _ in range(ws)]
        dist.all_gather(all_inputs, mine)
        # the reference arm prints on rank 0 only; other ranks exit 0 without work
        ref_rc, ref_out = None, None
        if rank != 0:
            buf = io.StringIO()
            with contextlib.redirect_stdout(buf):
                ref_rc = bench.run_reference(None)
            ref_out = buf.getvalue()
        dist.barrier()
        dist.destroy_process_group()
        q.put((rank, t_max, [t.tolist() for t in all_inputs], ref_rc, ref_out))
    except Exception as e:  # reported to the parent
        q.put((rank, "error", repr(e), None, None))


def test_two_rank_replicas_over_gloo():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(ws):
        r = q.get(timeout=120)
        res[r[0]] = r
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(ws):
        assert res[r][1] != "error", res[r][2]
        assert res[r][1] == 15.0                      # max over ranks, seen by every rank
    inputs = res[0][2]
    assert inputs == res[1][2]
    # no two ranks share a weight-copy seed or a token batch
    assert inputs[0][0] != inputs[1][0]
    assert not set(inputs[0][1:]) & set(inputs[1][1:])
    assert res[1][3] == 0 and res[1][4] == ""


def test_job_throughput_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    # 2 ranks x 32 tokens x 100 steps over the slowest rank's 50 ms
    assert bench.job_throughput(2, 32, 100, 50.0) == pytest.approx(2 * 32 * 100 / 0.05)
    assert bench.job_throughput(1, 32, 100, 50.0) * 2 == bench.job_throughput(2, 32, 100, 50.0)
