"""Host-side multi-rank logic of the benchmark on CPU: two gloo ranks on
127.0.0.1.  Heads are independent, so ranks shard the batch with no
collective on the data path; the only collectives are the barrier and the
max over ranks of the step time that the whole-job throughput divides by."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    ws, r, local = bench.dist_setup()
    bench.barrier(ws)
    # rank r took (r + 1) ms for 1000 units: the job runs at the slowest rank
    value, ms = bench.whole_job_rate(1000, float(r + 1), ws, torch.device("cpu"))
    q.put((r, ws, value, ms))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for r, ws, value, ms in res:
        assert ws == 2
        assert ms == 2.0                              # max over ranks
        assert abs(value - 2 * 1000 / 0.002) < 1e-6   # both ranks' units / slowest time
