"""GPU parity of the sharded hard and soft ECC (euler_characteristic_curves_gb300/shard.py),
through the C ABI: every rank of a plan runs in turn on one GPU (virtual ranks) and their partials
meet in one buffer, which is what the all-reduce computes across GPUs. Compared with the oracle
(bit for bit for the hard ECC) and with the single-call library result."""
import numpy as np
import pytest
import torch

import oracle
from euler_characteristic_curves_gb300 import ecc, shard, synthetic
from tests import _oracle_pool

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("world", [1, 2, 3, 7])
def test_volume_slabs_over_virtual_ranks(world):
    v = synthetic.grf((40, 130, 260), seed=50, device=DEV)  # ragged tiles, TMA-staged kernel
    want = _oracle_pool.hard_volume(v.cpu().numpy(), 256, 0.0, 1.0)
    hist = torch.zeros(256, dtype=torch.int64, device=DEV)
    for r, (a, b) in enumerate(shard.slab_plan(v.shape[0], world)):
        shard.volume_partial(v[a:b + 1], 256, 0.0, 1.0, r, hist)
    ecc.hist_to_curve(hist)
    np.testing.assert_array_equal(hist.cpu().numpy(), want)
    # the one-call path of a single rank gives the same curve
    if world == 1:
        got = shard.ecc_hard_volume_sharded(v, 256, 0.0, 1.0, 0)
        np.testing.assert_array_equal(got.cpu().numpy(), want)


def test_uint8_volume_and_1024cube_over_virtual_ranks():
    q = synthetic.quantise_u8(synthetic.grf((33, 70, 300), seed=51, device=DEV))
    hist = torch.zeros(256, dtype=torch.int64, device=DEV)
    for r, (a, b) in enumerate(shard.slab_plan(q.shape[0], 4)):
        shard.volume_partial(q[a:b + 1], 256, 0.0, 255.0, r, hist)
    ecc.hist_to_curve(hist)
    np.testing.assert_array_equal(hist.cpu().numpy(),
                                  oracle.ecc_hard(q.cpu().numpy(), 256, 0.0, 255.0))
    # the benchmark volume over four ranks equals the one-call curve (checked against the oracle
    # in test_workload_1024cube_f32)
    v = synthetic.grf((1024, 1024, 1024), seed=4, device=DEV)
    hist = torch.zeros(256, dtype=torch.int64, device=DEV)
    for r, (a, b) in enumerate(shard.slab_plan(1024, 4)):
        shard.volume_partial(v[a:b + 1], 256, 0.0, 1.0, r, hist)
    ecc.hist_to_curve(hist)
    assert torch.equal(hist, ecc.ecc_hard(v.unsqueeze(0), 256, 0.0, 1.0)[0])


def test_batch_over_virtual_ranks():
    imgs = torch.from_numpy(synthetic.grf((200, 333), seed=52, batch=7)).to(DEV)
    want = oracle.ecc_hard(imgs.cpu().numpy(), 100, 0.0, 1.0, ndim=2)
    for world in (2, 3):
        hist = torch.zeros((7, 100), dtype=torch.int64, device=DEV)
        for lo, hi in shard.batch_plan(7, world):
            ecc.ecc_hard_partial(imgs[lo:hi], 100, 0.0, 1.0, hist[lo:hi], ndim=2)
        ecc.hist_to_curve(hist)
        np.testing.assert_array_equal(hist.cpu().numpy(), want)


def test_soft_batch_over_virtual_ranks():
    img = synthetic.grf((64, 96), seed=53, batch=5)
    tau = synthetic.uniform_thresholds(32)
    u = synthetic.soft_direction(2, seed=54)
    g = synthetic.upstream_grad((5, 32), seed=55)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    x, t, uu, gg, alpha = d(img), d(tau), d(u), d(g), torch.ones(1, device=DEV)
    ref_s = oracle.ecc_soft_fwd(img, tau, 50.0, 1.0, u, ndim=2)
    ref = oracle.ecc_soft_bwd(img, tau, 50.0, 1.0, u, g, ndim=2, want_img=False)
    for world in (1, 2, 3):
        parts = []
        for lo, hi in shard.batch_plan(5, world):
            bufs = []
            shard.soft_ecc_batch_sharded(x[lo:hi], lo, 5, t, 50.0, alpha, uu, gg[lo:hi],
                                         allreduce=lambda b: bufs.append(b.clone()))
            parts.append(bufs[0])
        total = torch.stack(parts).sum(0).double().cpu().numpy()
        S, tail = total[:5 * 32].reshape(5, 32), total[5 * 32:]
        tol = lambda want: 1e-6 + 1e-4 * np.abs(want)
        assert np.all(np.abs(S - ref_s) <= tol(ref_s))
        assert np.all(np.abs(tail[:32] - ref["grad_tau"]) <= 2 * tol(ref["grad_tau"]))
        assert abs(tail[32] - ref["grad_alpha"]) <= 2 * tol(ref["grad_alpha"])
        assert np.all(np.abs(tail[33:] - ref["grad_u"]) <= 2 * tol(ref["grad_u"]))


def test_partial_signs_cancel_and_accumulate():
    """+1 then -1 of the same image leaves the histogram unchanged, and a partial adds to what the
    histogram holds (it is not zeroed)."""
    v = torch.from_numpy(synthetic.grf((20, 44, 132), seed=56)).to(DEV)
    h = torch.full((64,), 5, dtype=torch.int64, device=DEV)
    ecc.ecc_hard_partial(v, 64, 0.0, 1.0, h, sign=1, ndim=3)
    ecc.ecc_hard_partial(v, 64, 0.0, 1.0, h, sign=-1, ndim=3)
    assert torch.all(h == 5)
    ecc.ecc_hard_partial(v, 64, 0.0, 1.0, h, sign=1, ndim=3)
    ecc.hist_to_curve(h)
    want = oracle.ecc_hard(v.cpu().numpy(), 64, 0.0, 1.0) + 5 * np.arange(1, 65)
    np.testing.assert_array_equal(h.cpu().numpy(), want)
