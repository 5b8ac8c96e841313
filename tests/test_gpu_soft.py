"""GPU parity for the soft ECC forward and backward against the fp64 oracle.

2-D images and 3-D volumes (the volume tests sit at the end). Tolerance (per element), for S,
grad_tau, grad_alpha and grad_u:
    |gpu - oracle| <= 1e-6 + 1e-4 |oracle|.
grad_img (an optional output) sums K terms per pixel that can cancel; its bound adds a term
proportional to the sum of the magnitudes of those terms (returned by the oracle):
    |gpu - oracle| <= 1e-6 + 1e-4 |oracle| + 4e-6 * sum|terms|.
"""
import numpy as np
import pytest
import torch

import oracle
from euler_characteristic_curves_gb300 import ecc, synthetic
from tests import _oracle_pool

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
RTOL, ATOL = 1e-4, 1e-6


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def assert_close(got, want, what, extra=None):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    tol = ATOL + RTOL * np.abs(want)
    if extra is not None:
        tol = tol + extra
    err = np.abs(got - want)
    bad = err > tol
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst "
                           f"err/tol = {np.max(err / tol):.3g}")
    return float(np.max(err / tol))


def run_both(img, tau, lam, alpha, u, g, want_img=True, sample=None):
    """GPU fwd + bwd through the C ABI, and the oracle (optionally only on sampled images)."""
    a = np.asarray([alpha], np.float32)
    s, ws = ecc.ecc_soft_fwd(dev(img), dev(tau), lam, dev(a), dev(u))
    res = ecc.ecc_soft_bwd(dev(img), dev(tau), lam, dev(a), dev(u), dev(g), ws,
                           want_img=want_img)
    s = s.cpu().numpy()
    res = {k: v.cpu().numpy() for k, v in res.items()}
    imgs = img if sample is None else img[sample]
    gs = g if sample is None else g[sample]
    nd = len(u)
    ref_s = oracle.ecc_soft_fwd(imgs, tau, lam, alpha, u, ndim=nd)
    ref = oracle.ecc_soft_bwd(imgs, tau, lam, alpha, u, gs, ndim=nd, want_img=want_img)
    return s, res, ref_s, ref


def compare(img, tau, lam, alpha, u, g, want_img=True):
    s, res, ref_s, ref = run_both(img, tau, lam, alpha, u, g, want_img)
    assert_close(s, ref_s, "S")
    assert_close(res["grad_tau"], ref["grad_tau"], "grad_tau")
    assert_close(res["grad_alpha"][0], ref["grad_alpha"], "grad_alpha")
    assert_close(res["grad_u"], ref["grad_u"], "grad_u")
    if want_img:
        assert_close(res["grad_img"], ref["grad_img"], "grad_img",
                     extra=4e-6 * ref["grad_img_absterms"])
    else:
        assert "grad_img" not in res


@pytest.mark.parametrize("shape,batch", [((1, 1), 1), ((1, 9), 2), ((7, 1), 1), ((5, 7), 3),
                                         ((33, 65), 2), ((64, 64), 1), ((100, 130), 2),
                                         ((31, 257), 1)])
def test_soft_parity_shapes(shape, batch):
    img = synthetic.grf(shape, seed=sum(shape), batch=batch) if min(shape) > 1 else \
        np.random.default_rng(1).random((batch,) + shape).astype(np.float32)
    K = 24
    tau = synthetic.uniform_thresholds(K, -0.2, 1.2)
    u = synthetic.soft_direction(2, seed=batch)
    g = synthetic.upstream_grad((batch, K), seed=3)
    compare(img, tau, 50.0, 1.0, u, g)


@pytest.mark.parametrize("K", [1, 7, 128, 129, 300])
def test_soft_parity_K(K):
    img = synthetic.grf((48, 80), seed=K, batch=2)
    rng = np.random.default_rng(K)
    tau = rng.uniform(-0.1, 1.1, size=K).astype(np.float32)  # unsorted thresholds
    u = synthetic.soft_direction(2, seed=K)
    g = synthetic.upstream_grad((2, K), seed=K + 1)
    compare(img, tau, 50.0, 1.0, u, g)


@pytest.mark.parametrize("shape,batch,K", [((1, 9), 2, 24), ((33, 65), 2, 24), ((48, 80), 1, 129),
                                           ((31, 257), 1, 300), ((2, 3, 4), 2, 24),
                                           ((9, 17, 33), 1, 129), ((12, 20, 45), 2, 300)])
def test_soft_parity_without_the_image_gradient(shape, batch, K):
    """The backward without an image gradient (the one a loss on S alone takes) keeps no
    per-pixel accumulator; threshold counts past one chunk of the backward (128) included."""
    img = synthetic.grf(shape, seed=sum(shape) + K, batch=batch) if min(shape) > 1 else \
        np.random.default_rng(K).random((batch,) + shape).astype(np.float32)
    tau = synthetic.uniform_thresholds(K, -0.2, 1.2)
    u = synthetic.soft_direction(len(shape), seed=K)
    g = synthetic.upstream_grad((batch, K), seed=K + 1)
    compare(img, tau, 50.0, 1.0, u, g, want_img=False)


@pytest.mark.parametrize("lam,alpha", [(1.0, 1.0), (5.0, -0.7), (50.0, 2.5), (500.0, 1.0),
                                       (3000.0, 0.3)])
def test_soft_parity_lambda_alpha(lam, alpha):
    img = synthetic.grf((57, 90), seed=int(lam), batch=2)
    tau = synthetic.uniform_thresholds(32, -1.0, 1.5)
    u = np.asarray([0.13, -0.21], np.float32)
    g = synthetic.upstream_grad((2, 32), seed=5)
    compare(img, tau, lam, alpha, u, g)


def test_soft_ties_and_zero_direction():
    q = synthetic.quantise_u8(synthetic.grf((60, 70), seed=6, batch=2)).astype(np.float32) / 255
    tau = synthetic.uniform_thresholds(40)
    g = synthetic.upstream_grad((2, 40), seed=7)
    compare(q, tau, 50.0, 1.0, np.zeros(2, np.float32), g)  # exact ties in X everywhere
    compare(q, tau, 50.0, 0.5, np.asarray([0.0, 0.3], np.float32), g)
    const = np.full((2, 20, 30), 0.25, np.float32)
    compare(const, tau, 50.0, 1.0, np.zeros(2, np.float32), g)


def test_soft_large_lambda_matches_hard():
    q = np.random.default_rng(8).integers(0, 6, size=(2, 40, 50)).astype(np.float32)
    tau = (np.arange(7) - 0.5).astype(np.float32)
    a = np.asarray([1.0], np.float32)
    s, _ = ecc.ecc_soft_fwd(dev(q), dev(tau), 1.0e4, dev(a), dev(np.zeros(2, np.float32)))
    hard = ecc.ecc_hard(dev(q), 7, -0.5, 5.5, ndim=2).cpu().numpy()
    np.testing.assert_allclose(s.cpu().numpy(), hard.astype(np.float64), atol=1e-6)


def test_autograd_layer_matches_direct_calls():
    img = synthetic.grf((40, 50), seed=9, batch=2)
    tau = dev(synthetic.uniform_thresholds(16)).requires_grad_()
    alpha = torch.ones(1, device=DEV, requires_grad=True)
    u = dev(np.asarray([0.05, -0.08], np.float32)).requires_grad_()
    x = dev(img).requires_grad_()
    g = dev(synthetic.upstream_grad((2, 16), seed=10))
    s = ecc.soft_ecc(x, tau, alpha, u, 50.0)
    (s * g).sum().backward()
    s2, ws = ecc.ecc_soft_fwd(dev(img), tau.detach(), 50.0, alpha.detach(), u.detach())
    res = ecc.ecc_soft_bwd(dev(img), tau.detach(), 50.0, alpha.detach(), u.detach(), g, ws,
                           want_img=True)
    assert torch.equal(s.detach(), s2)
    assert torch.equal(tau.grad, res["grad_tau"])
    assert torch.equal(alpha.grad, res["grad_alpha"])
    assert torch.equal(u.grad, res["grad_u"])
    assert torch.equal(x.grad, res["grad_img"])


def test_workload_64x256sq_soft():
    """The benchmark workload at full size: 64 GRF images 256^2, K = 128 thresholds on [0, 1],
    lambda = 50, alpha = 1, u ~ N(0, 0.1^2), upstream dL/dS ~ N(0, 1) on every image. The oracle
    runs on all 64 images (one process per host core) and every output is compared element by
    element: S, grad_tau, grad_alpha, grad_u and grad_img. For grad_img the test also reports how
    far inside its documented bound the kernels land (worst err/tol with and without the
    cancellation term)."""
    img = synthetic.grf((256, 256), seed=6, batch=64)
    tau = synthetic.uniform_thresholds(128)
    u = synthetic.soft_direction(2, seed=7)
    g = synthetic.upstream_grad((64, 128), seed=8)
    a = np.asarray([1.0], np.float32)
    s, ws = ecc.ecc_soft_fwd(dev(img), dev(tau), 50.0, dev(a), dev(u))
    res = ecc.ecc_soft_bwd(dev(img), dev(tau), 50.0, dev(a), dev(u), dev(g), ws, want_img=True)
    s = s.cpu().numpy()
    res = {k: v.cpu().numpy() for k, v in res.items()}
    ref_s, ref = _oracle_pool.soft_batch(img, tau, 50.0, 1.0, u, g, ndim=2, want_img=True)
    assert_close(s, ref_s, "S")
    assert_close(res["grad_tau"], ref["grad_tau"], "grad_tau")
    assert_close(res["grad_alpha"][0], ref["grad_alpha"], "grad_alpha")
    assert_close(res["grad_u"], ref["grad_u"], "grad_u")
    extra = 4e-6 * ref["grad_img_absterms"]
    worst = assert_close(res["grad_img"], ref["grad_img"], "grad_img", extra=extra)
    err = np.abs(res["grad_img"].astype(np.float64) - ref["grad_img"])
    plain = np.max(err / (ATOL + RTOL * np.abs(ref["grad_img"])))
    print(f"grad_img 64x256^2: worst err/tol {worst:.3g} (bound with the cancellation term), "
          f"{plain:.3g} against 1e-6 + 1e-4 |ref| alone")


# ---------------------------------------------------------------------------------------------
# 3-D volumes (3 x 3 x 3 neighbourhoods; tiles of 8 x 8 x 32 voxels)
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("shape,batch", [((1, 1, 1), 1), ((2, 3, 4), 2), ((1, 5, 70), 1),
                                         ((5, 1, 1), 1), ((9, 10, 33), 1), ((17, 9, 40), 2),
                                         ((8, 8, 32), 1), ((20, 19, 65), 1)])
def test_soft3d_parity_shapes(shape, batch):
    """Shapes below, at and across the tile edges along each axis, with ragged tails."""
    img = synthetic.grf(shape, seed=sum(shape), batch=batch) if min(shape) > 1 else \
        np.random.default_rng(2).random((batch,) + shape).astype(np.float32)
    K = 20
    tau = synthetic.uniform_thresholds(K, -0.3, 1.3)
    u = synthetic.soft_direction(3, seed=batch + 10)
    g = synthetic.upstream_grad((batch, K), seed=4)
    compare(img, tau, 50.0, 1.0, u, g)


@pytest.mark.parametrize("K,lam,alpha", [(1, 50.0, 1.0), (129, 50.0, 1.0), (33, 2.0, -0.6),
                                         (33, 800.0, 1.7), (16, 4000.0, 0.4)])
def test_soft3d_parity_K_lambda_alpha(K, lam, alpha):
    img = synthetic.grf((12, 14, 36), seed=K, batch=2)
    rng = np.random.default_rng(K + 1)
    tau = rng.uniform(-0.4, 1.4, size=K).astype(np.float32)  # unsorted thresholds
    u = np.asarray([0.11, -0.17, 0.07], np.float32)
    g = synthetic.upstream_grad((2, K), seed=K + 2)
    compare(img, tau, lam, alpha, u, g)


def test_soft3d_ties_and_zero_direction():
    q = synthetic.quantise_u8(synthetic.grf((10, 12, 40), seed=11, batch=2)).astype(np.float32)
    q /= 255
    tau = synthetic.uniform_thresholds(24)
    g = synthetic.upstream_grad((2, 24), seed=12)
    compare(q, tau, 50.0, 1.0, np.zeros(3, np.float32), g)  # exact ties in X everywhere
    compare(q, tau, 50.0, 0.5, np.asarray([0.0, 0.0, 0.3], np.float32), g)
    const = np.full((2, 9, 9, 33), 0.25, np.float32)
    compare(const, tau, 50.0, 1.0, np.zeros(3, np.float32), g)


def test_soft3d_large_lambda_matches_hard():
    q = np.random.default_rng(13).integers(0, 6, size=(2, 11, 12, 37)).astype(np.float32)
    tau = (np.arange(7) - 0.5).astype(np.float32)
    a = np.asarray([1.0], np.float32)
    s, _ = ecc.ecc_soft_fwd(dev(q), dev(tau), 1.0e4, dev(a), dev(np.zeros(3, np.float32)))
    hard = ecc.ecc_hard(dev(q), 7, -0.5, 5.5, ndim=3).cpu().numpy()
    np.testing.assert_allclose(s.cpu().numpy(), hard.astype(np.float64), atol=1e-6)


def test_soft3d_autograd_layer():
    img = synthetic.grf((10, 16, 40), seed=14, batch=2)
    tau = dev(synthetic.uniform_thresholds(16)).requires_grad_()
    alpha = torch.ones(1, device=DEV, requires_grad=True)
    u = dev(np.asarray([0.05, -0.08, 0.02], np.float32)).requires_grad_()
    x = dev(img).requires_grad_()
    g = dev(synthetic.upstream_grad((2, 16), seed=15))
    s = ecc.soft_ecc(x, tau, alpha, u, 50.0)
    (s * g).sum().backward()
    ref = oracle.ecc_soft_bwd(img, tau.detach().cpu().numpy(), 50.0, 1.0,
                              u.detach().cpu().numpy(), g.cpu().numpy(), ndim=3)
    assert_close(tau.grad.cpu().numpy(), ref["grad_tau"], "grad_tau")
    assert_close(u.grad.cpu().numpy(), ref["grad_u"], "grad_u")
    assert_close(x.grad.cpu().numpy(), ref["grad_img"], "grad_img",
                 extra=4e-6 * ref["grad_img_absterms"])


def test_soft3d_volume_64cubed_sampled():
    """A larger volume batch (8 x 64^3, 64 tiles each): S on two sampled volumes, and every
    gradient with the upstream gradient non-zero on those volumes only."""
    img = synthetic.grf((64, 64, 64), seed=16, batch=8)
    tau = synthetic.uniform_thresholds(64)
    u = synthetic.soft_direction(3, seed=17)
    g_full = synthetic.upstream_grad((8, 64), seed=18)
    sample = np.asarray([0, 5])
    g = np.zeros_like(g_full)
    g[sample] = g_full[sample]
    s, res, ref_s, ref = run_both(img, tau, 50.0, 1.0, u, g, want_img=True, sample=sample)
    assert_close(s[sample], ref_s, "S")
    assert_close(res["grad_tau"], ref["grad_tau"], "grad_tau")
    assert_close(res["grad_alpha"][0], ref["grad_alpha"], "grad_alpha")
    assert_close(res["grad_u"], ref["grad_u"], "grad_u")
    assert_close(res["grad_img"][sample], ref["grad_img"], "grad_img",
                 extra=4e-6 * ref["grad_img_absterms"])


@pytest.mark.parametrize("shape,batch,ndim", [((70, 130), 3, 2), ((12, 20, 45), 2, 3)])
def test_soft_stats_counts_the_contributing_voxels(shape, batch, ndim):
    """stats[0] = voxels with c_X != 0. The oracle's image gradient is lambda c_X sum_k g_k w_k
    per voxel: a random upstream gradient makes it clearly non-zero exactly there, while where
    c_X = 0 the oracle's per-cell sum leaves only rounding residue (below 1e-9 of the sum of the
    magnitudes of its terms), which gives the expected count."""
    img = synthetic.grf(shape, seed=21, batch=batch)
    K = 16
    tau = synthetic.uniform_thresholds(K)
    u = synthetic.soft_direction(ndim, seed=22)
    g = synthetic.upstream_grad((batch, K), seed=23)
    a = np.asarray([1.0], np.float32)
    # c_X depends on the order of X only, not on lambda: one oracle run at a lambda where no
    # sigmoid derivative underflows gives the count for both launches
    ref = oracle.ecc_soft_bwd(img, tau, 50.0, 1.0, u, g, ndim=ndim)
    for lam, direct in ((50.0, False), (4000.0, True)):
        _, ws = ecc.ecc_soft_fwd(dev(img), dev(tau), lam, dev(a), dev(u))
        st = ecc.ecc_soft_stats(dev(img), K, ws, ndim=ndim).cpu().numpy()
        assert st[0] == np.count_nonzero(np.abs(ref["grad_img"]) >
                                          1e-9 * ref["grad_img_absterms"])
        tile = (64, 32) if ndim == 2 else (32, 8, 8)
        tiles = batch * int(np.prod([-(-n // t) for n, t in zip(shape[::-1], tile)]))
        assert st[2] == tiles
        assert (st[1] > 0) == direct


@pytest.mark.parametrize("ndim", [2, 3])
def test_dense_critical_lists(ndim):
    """Inputs where most voxels contribute: a checkerboard (with a tiny ramp so that no two values
    tie) and white noise. Every tile's list is then far longer than one staging chunk, so the
    forward and backward walk many chunks and groups per tile; the whole curve and every gradient
    must still match the oracle."""
    shape = (64, 128) if ndim == 2 else (16, 16, 64)
    idx = np.indices(shape)
    cb = (idx.sum(0) % 2).astype(np.float64)
    ramp = np.arange(int(np.prod(shape)), dtype=np.float64).reshape(shape) / np.prod(shape)
    noise = np.random.default_rng(31).random(shape)
    img = np.stack([0.5 * cb + 0.4 * ramp, noise]).astype(np.float32)
    K = 64
    tau = synthetic.uniform_thresholds(K)
    u = (synthetic.soft_direction(ndim, seed=32) * 0.1).astype(np.float32)
    g = synthetic.upstream_grad((2, K), seed=33)
    a = np.asarray([1.0], np.float32)
    _, ws = ecc.ecc_soft_fwd(dev(img), dev(tau), 50.0, dev(a), dev(u))
    st = ecc.ecc_soft_stats(dev(img), K, ws, ndim=ndim).cpu().numpy()
    assert st[0] > 0.4 * img.size  # dense lists: most voxels contribute
    compare(img, tau, 50.0, 1.0, u, g)


def test_soft_at_the_largest_K():
    """K = 8192 (ECC_MAX_K): 64 threshold passes per tile in the forward and backward, spread
    over a range wider than the data, so thresholds sit on both sides of every value.

    S, grad_alpha, grad_u and grad_img are held to the bounds of the other tests. Among 8192
    grad_tau entries some are sums whose terms cancel to a thousandth of their size; those are
    held, like grad_img, to the plain bound plus 4e-6 times the sum of |terms| (the oracle's
    grad_tau_absterms), and every other entry to the plain bound."""
    img = synthetic.grf((9, 21), 51, batch=2)
    tau = np.linspace(-0.25, 1.25, 8192).astype(np.float32)
    g = synthetic.upstream_grad((2, 8192), seed=52)
    u = np.asarray([0.03, -0.02], np.float32)
    s, res, ref_s, ref = run_both(img, tau, 50.0, 1.0, u, g)
    assert_close(s, ref_s, "S")
    assert_close(res["grad_alpha"][0], ref["grad_alpha"], "grad_alpha")
    assert_close(res["grad_u"], ref["grad_u"], "grad_u")
    assert_close(res["grad_img"], ref["grad_img"], "grad_img",
                 extra=4e-6 * ref["grad_img_absterms"])
    gt, rt, ab = res["grad_tau"], ref["grad_tau"], ref["grad_tau_absterms"]
    worst = assert_close(gt, rt, "grad_tau", extra=4e-6 * ab)
    plain = np.abs(gt - rt) > ATOL + RTOL * np.abs(rt)
    cancelled = np.abs(rt) < 1e-2 * ab  # sums cancelled to under a hundredth of their terms
    print(f"grad_tau: worst err/tol {worst:.3g} of the cancellation-aware bound; "
          f"{plain.sum()} of {plain.size} outside the plain bound")
    assert not (plain & ~cancelled).any()


def test_soft_at_the_largest_batch():
    """65535 images (the grid's y extent holds one (image, direction) pair each), 2 x 3 pixels,
    every image different; forward and backward against the oracle over the whole batch."""
    rng = np.random.default_rng(53)
    img = rng.random((65535, 2, 3)).astype(np.float32)
    tau = synthetic.uniform_thresholds(5)
    g = rng.standard_normal((65535, 5)).astype(np.float32)
    compare(img, tau, 20.0, 1.0, np.asarray([0.1, 0.05], np.float32), g, want_img=False)
