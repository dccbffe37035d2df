"""The bench's multi-GPU logic (replicas, no data-path collective) with two ranks on the
CPU over gloo: rendezvous at 127.0.0.1, the barrier, the max-over-ranks step time, the
whole-job aggregate, and the reference arm doing no work on ranks other than 0."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "LOCAL_RANK": str(rank), "WORLD_SIZE": str(ws)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    got_ws, got_rank, local = bench.dist_setup(backend="gloo")
    bench.barrier(got_ws)
    # each replica "measured" a different step time; the job is as slow as the slowest
    t_ms = bench.max_over_ranks(100.0 + 10.0 * rank, got_ws, device="cpu")
    value = bench.job_tok_s(got_ws, t_ms)
    # the reference arm: rank 0 alone runs it; the other ranks return at once
    ref_rc = None
    if rank != 0:
        class A:
            warmup, steps = 1, 1
        ref_rc = bench.run_reference(A())
    bench.barrier(got_ws)
    dist.destroy_process_group()
    q.put((rank, got_ws, got_rank, local, t_ms, value, ref_rc))


def test_two_ranks_gloo():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got_ws, got_rank, local, t_ms, value, ref_rc in results:
        assert (got_ws, got_rank, local) == (ws, rank, rank)
        assert t_ms == 110.0                              # max over ranks, identical on both
        assert abs(value - 2 * 3314 / 0.110) < 1e-6       # whole-job tokens over the slowest step
        if rank != 0:
            assert ref_rc == 0
