"""The bench's N>1 path on CPU with gloo, world size 2: each rank is an
independent replica; the only collective is the max over ranks of the timed
region, and the reference arm runs on rank 0 alone."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    got = bench.max_over_ranks(10.0 + 5.0 * rank, world)
    env = bench.dist_env()
    # the reference arm: every rank but 0 returns at once without work
    rc = bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "1"])) if rank == 1 else None
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, got, env, rc))


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [15.0, 15.0]
    assert res[0][2] == (2, 0, 0) and res[1][2] == (2, 1, 1)
    assert res[1][3] == 0
