"""Multi-process logic on CPU (gloo, world size 2), no GPU.

* bench.py's timing aggregation: every rank reports its time and the slowest one is taken.
* The sharding module (euler_characteristic_curves_gb300/shard.py) end to end over two ranks:
  its slab and batch plans, its per-rank bookkeeping (which rank subtracts the shared plane,
  where a rank's rows go) and its one all-reduce. The per-rank compute that the CUDA library does
  on a GPU is injected here as the oracle on CPU tensors (the histogram is the oracle curve's
  first difference), so the test checks the plan and the exchange against the oracle's curve of
  the whole grid, bit for bit for the hard ECC.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

WORLD = 2
NB = 40


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def oracle_partial(x, nbins, vmin, vmax, sign, hist, ndim):
    """The library's ecc_hard_partial restated with the oracle: hist += sign * (per-bin counts)."""
    import oracle

    curve = oracle.ecc_hard(x.numpy(), nbins, vmin, vmax, ndim=ndim)
    h = np.diff(curve, axis=-1, prepend=0).astype(np.int64)
    hist += sign * torch.from_numpy(h).view(hist.shape)


def cumsum_(hist):
    hist.copy_(torch.cumsum(hist, dim=-1))


def oracle_soft_local(images, tau, lam, alpha, u, grad_out, ndim):
    import oracle

    img = images.numpy()
    s = oracle.ecc_soft_fwd(img, tau.numpy(), lam, float(alpha[0]), u.numpy(), ndim=ndim)
    r = oracle.ecc_soft_bwd(img, tau.numpy(), lam, float(alpha[0]), u.numpy(),
                            grad_out.numpy(), ndim=ndim, want_img=False)
    f = lambda a: torch.as_tensor(np.asarray(a, np.float64)).float()
    return f(s), (f(r["grad_tau"]), f([r["grad_alpha"]]), f(r["grad_u"]))


def _worker(rank, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        import bench
        from euler_characteristic_curves_gb300 import shard, synthetic

        slowest = bench.max_over_ranks(1.5 + rank, WORLD)

        vol = torch.from_numpy(synthetic.grf((14, 12, 13), seed=31))
        a, b = shard.slab_plan(vol.shape[0], WORLD)[rank]
        curve = shard.ecc_hard_volume_sharded(vol[a:b + 1].contiguous(), NB, 0.0, 1.0, rank,
                                              partial=oracle_partial, to_curve=cumsum_)

        imgs = torch.from_numpy(synthetic.grf((9, 11), seed=32, batch=5))
        lo, hi = shard.batch_plan(5, WORLD)[rank]
        bcurve = shard.ecc_hard_batch_sharded(imgs[lo:hi].contiguous(), lo, 5, NB, 0.0, 1.0, 2,
                                              partial=oracle_partial, to_curve=cumsum_)

        simg = torch.from_numpy(synthetic.grf((8, 10), seed=33, batch=3))
        tau = torch.from_numpy(synthetic.uniform_thresholds(12))
        u = torch.tensor([0.05, -0.1])
        g = torch.from_numpy(synthetic.upstream_grad((3, 12), seed=34))
        lo, hi = shard.batch_plan(3, WORLD)[rank]
        S, grads = shard.soft_ecc_batch_sharded(simg[lo:hi].contiguous(), lo, 3, tau, 20.0,
                                                torch.ones(1), u, g[lo:hi].contiguous(),
                                                local=oracle_soft_local)
        q.put((rank, slowest, curve.tolist(), bcurve.tolist(), S.tolist(),
               [t.tolist() for t in grads]))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_rank_sharding_through_the_module():
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
    full = oracle.ecc_hard(vol, NB, 0.0, 1.0).tolist()
    batch = oracle.ecc_hard(synthetic.grf((9, 11), seed=32, batch=5), NB, 0.0, 1.0,
                            ndim=2).tolist()
    simg = synthetic.grf((8, 10), seed=33, batch=3)
    tau = synthetic.uniform_thresholds(12)
    g = synthetic.upstream_grad((3, 12), seed=34)
    u = np.asarray([0.05, -0.1], np.float32)
    ref_s = oracle.ecc_soft_fwd(simg, tau, 20.0, 1.0, u, ndim=2)
    ref = oracle.ecc_soft_bwd(simg, tau, 20.0, 1.0, u, g, ndim=2, want_img=False)
    for rank, slowest, curve, bcurve, S, grads in results:
        assert slowest == 2.5
        assert curve == full  # every rank holds the whole volume's curve
        assert bcurve == batch
        np.testing.assert_allclose(np.asarray(S), ref_s, rtol=1e-5, atol=1e-6)
        np.testing.assert_allclose(grads[0], ref["grad_tau"], rtol=1e-5, atol=1e-5)
        np.testing.assert_allclose(grads[1][0], ref["grad_alpha"], rtol=1e-5, atol=1e-5)
        np.testing.assert_allclose(grads[2], ref["grad_u"], rtol=1e-5, atol=1e-5)


def test_slab_and_batch_plans():
    """Slabs cover the volume, consecutive slabs share exactly one plane, their lengths differ by
    at most one; batch ranges tile the batch."""
    from euler_characteristic_curves_gb300 import shard

    for depth in (1, 2, 3, 7, 64, 1024):
        for world in (1, 2, 3, 4, 8, 9):
            plan = shard.slab_plan(depth, world)
            assert len(plan) == world and plan[0][0] == 0 and plan[-1][1] == depth - 1
            for (a0, b0), (a1, b1) in zip(plan[:-1], plan[1:]):
                assert b0 == a1 and a0 <= b0
            spans = [b - a for a, b in plan]
            assert max(spans) - min(spans) <= 1
    for batch in (1, 5, 64):
        for world in (1, 2, 3, 8):
            plan = shard.batch_plan(batch, world)
            assert plan[0][0] == 0 and plan[-1][1] == batch
            assert all(h0 == l1 for (_, h0), (l1, _) in zip(plan[:-1], plan[1:]))


def test_virtual_ranks_on_cpu_match_the_oracle():
    """The slab identity through the module with every rank in one process (their partials summed
    into one histogram), for several world sizes, single-plane slabs included."""
    import oracle
    from euler_characteristic_curves_gb300 import shard, synthetic

    vol = torch.from_numpy(synthetic.grf((9, 10, 11), seed=35))
    want = oracle.ecc_hard(vol.numpy(), NB, 0.0, 1.0)
    for world in (1, 2, 3, 8, 12):
        hist = torch.zeros(NB, dtype=torch.int64)
        for r, (a, b) in enumerate(shard.slab_plan(vol.shape[0], world)):
            shard.volume_partial(vol[a:b + 1].contiguous(), NB, 0.0, 1.0, r, hist,
                                 partial=oracle_partial)
        cumsum_(hist)
        np.testing.assert_array_equal(hist.numpy(), want)
