"""The N-GPU launch path of bench.py on CPU: two ranks over gloo.

With more than one rank every rank runs an independent replica of the
workload (the path shards over (row, KV head) with no exchange step, so no
collective touches the data path); the ranks meet only at the barriers around
the timed region and at the max-over-ranks of the timings.  The reference arm
runs on rank 0 alone.
"""
import os
import socket
import sys

import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    ws, r, local = bench._dist()
    assert (ws, r, local) == (world, rank, rank) and dist.get_backend() == "gloo"
    bench._barrier(ws)
    t_max = bench._max_over_ranks(1.0 + rank, ws)           # each rank's own timing
    args = type("A", (), {"workload": "tiny", "seq_len": None, "bits": None, "steps": 1, "warmup": 3})()
    ref = bench.run_reference(args, ws, r) if r != 0 else "rank 0 runs the oracle"
    bench._barrier(ws)
    out.put((rank, t_max, ref))
    dist.destroy_process_group()


def test_two_ranks_over_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [t for _, t, _ in res] == [2.0, 2.0]      # every rank reports the slowest rank's time
    assert res[1][2] is None                         # the reference arm does no work off rank 0
