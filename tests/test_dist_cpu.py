"""Multi-process logic on CPU (gloo, world size 2), no GPU.

* bench.py's timing aggregation: every rank reports its time and the slowest one is taken.
* Sharding one volume over ranks: slabs that overlap by one plane, each rank computing its slab's
  curve; the global curve is the allreduce-sum of the slab curves minus the curves of the shared
  planes (inclusion-exclusion for the Euler characteristic). The per-slab curves come from the
  oracle here, so the test checks the exchange logic, not the kernels.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        import bench
        import oracle
        from euler_characteristic_curves_gb300 import synthetic

        slowest = bench.max_over_ranks(1.5 + rank, WORLD)

        vol = synthetic.grf((14, 12, 13), seed=31)
        D = vol.shape[0]
        cut = D // 2  # rank 0: planes [0, cut], rank 1: [cut, D); plane `cut` is shared
        lo, hi = (0, cut + 1) if rank == 0 else (cut, D)
        curve = oracle.ecc_hard(vol[lo:hi], 40, 0.0, 1.0).astype(np.int64)
        if rank == 0:
            curve = curve - oracle.ecc_hard(vol[cut], 40, 0.0, 1.0)
        t = torch.from_numpy(curve)
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        q.put((rank, slowest, t.numpy().tolist()))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_rank_timing_max_and_slab_sharding():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    results = [q.get(timeout=240) for _ in range(WORLD)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    import oracle
    from euler_characteristic_curves_gb300 import synthetic

    vol = synthetic.grf((14, 12, 13), seed=31)
    full = oracle.ecc_hard(vol, 40, 0.0, 1.0).tolist()
    for rank, slowest, curve in results:
        assert slowest == 2.5
        assert curve == full
