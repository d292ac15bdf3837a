"""The multi-GPU path of bench.py on the CPU: replicas only, two ranks over gloo.

Canvases are independent, so N GPUs run N replicas with disjoint canvas seeds
and no data-path collective; the only collectives are the barrier around the
timed region and the max over ranks of the timed seconds.  This runs the
bench's own helpers (seeding, barrier, max-reduction, whole-job rate) in two
processes joined by a gloo process group at 127.0.0.1.
"""
import os
import socket

import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, local = bench.dist_setup()
    seconds = 1.5 + rank  # the slower rank sets the job's time
    bench.barrier(w)
    slowest = bench.reduce_max(seconds, w)
    rate = bench.whole_job_rate(256, 10, w, slowest)
    out.put((r, w, local, bench.replica_seeds(r, 4), slowest, rate))
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_replicas_over_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    seeds = [set(r[3]) for r in res]
    assert [r[0] for r in res] == [0, 1] and all(r[1] == world and r[2] == r[0] for r in res)
    assert seeds[0].isdisjoint(seeds[1]) and len(seeds[0] | seeds[1]) == 8
    # every rank sees the slowest rank's time and the same whole-job rate: 2 ranks x 10 steps x 256 / 2.5 s
    assert all(r[4] == 2.5 for r in res)
    assert all(abs(r[5] - 2 * 10 * 256 / 2.5) < 1e-9 for r in res)

