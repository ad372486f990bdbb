"""The multi-GPU path runs independent replicas (one per rank): the whole-job
numbers are the committed tokens summed over the ranks and the slowest rank's
time. Checked here with two gloo ranks on the CPU."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r committed 10 + r tokens in 100 + 7r ms; end to end 20 + r tokens in 2 + r s
    out = bench.aggregate_replicas(10 + rank, 100.0 + 7 * rank, 20 + rank, 2.0 + rank, "cpu")
    q.put((rank, out))
    dist.barrier()
    dist.destroy_process_group()


def test_replica_totals_sum_tokens_and_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        assert got[r] == (21.0, 107.0, 41.0, 3.0)
