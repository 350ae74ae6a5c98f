"""bench.py's multi-rank plumbing on CPU: two gloo ranks rendezvous, meet at the barrier and
agree on the max-over-ranks time; the reference arm prints only on rank 0.  (The path itself
is replicas only: every rank runs an independent request; no data-path collective exists.)"""

import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, results):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    r, w, local = bench.dist_init()
    bench.dist_barrier(w)
    m = bench.dist_max(10.0 * (rank + 1) + 0.5, w)
    args = type("A", (), {"workload": "toy_q8_0", "warmup": 0, "steps": 1})()
    ref = bench.run_reference(args, r, w) if rank == 1 else "skipped"
    bench.dist_barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()
    results[rank] = (r, w, local, m, ref)


def test_two_gloo_ranks():
    port = _free_port()
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_rank_main, args=(2, port, results), nprocs=2, join=True)
        res = dict(results)
    assert res[0][:3] == (0, 2, 0) and res[1][:3] == (1, 2, 1)
    assert res[0][3] == res[1][3] == 20.5
    assert res[1][4] is None   # only rank 0 runs and prints the reference arm
