"""Multi-rank path of bench.py on CPU: N independent replicas (one per rank) report the whole-job
throughput from the slowest rank's time. world_size 2 over gloo, rendezvous on 127.0.0.1."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed = [100.0, 250.0][rank]
    ms, tok = bench.aggregate_replicas(elapsed, world, 32, 10, torch.device("cpu"))
    dist.barrier()
    q.put((rank, ms, tok))
    dist.destroy_process_group()


def test_two_replicas_take_max_time_and_sum_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, tok in res:
        assert ms == 250.0
        assert abs(tok - 2 * 32 * 10 / 0.25) < 1e-9
