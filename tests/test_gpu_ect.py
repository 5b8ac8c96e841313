"""GPU parity for the soft Euler characteristic transform (several directions in one pass)
against the fp64 oracle, which evaluates the pinned single-direction soft ECC per direction.

Tolerances as in test_gpu_soft.py: |gpu - oracle| <= 1e-6 + 1e-4 |oracle| for S, grad_tau and
grad_alpha; grad_img (a sum over directions and thresholds that can cancel) adds
4e-6 * sum|terms|. grad_u[j, d] = sum_p dX_p x_{p,d} sums tens of thousands of voxels whose
terms cancel, so a small component cannot be reproduced to 1e-4 of itself by fp32 terms; its
bound adds the per-voxel allowance of grad_img carried through that sum. The per-voxel errors
come from separate fp32 sums, so they combine in quadrature:
    4e-6 * sqrt(sum_p (absterms_{j,p} |x_{p,d}|)^2),
with absterms_j the oracle's sum of |terms| of dX_p for direction j.
"""
import numpy as np
import pytest
import torch

import oracle
from euler_characteristic_curves_gb300 import ecc, synthetic

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


def directions(n, ndim, seed):
    U = (0.15 * np.random.default_rng(seed).standard_normal((n, ndim))).astype(np.float32)
    U[0] = 0.0  # the plain soft ECC of alpha f
    if n > 2:
        U[2] = -U[1]  # opposite directions
    return U


def axis_coords(n):
    """x_d(i) = (2 i - (n - 1)) / (n - 1), 0 on an axis of extent 1."""
    if n == 1:
        return np.zeros(1)
    return (2.0 * np.arange(n) - (n - 1)) / (n - 1)


def grad_u_allowance(img, tau, lam, alpha, U, g, ndim):
    """4e-6 * sqrt(sum_p (absterms_{j,p} |x_{p,d}|)^2) per direction j and axis d (see the
    module doc)."""
    shape = img.shape[-ndim:]
    out = np.zeros(U.shape, np.float64)
    for j in range(U.shape[0]):
        ab = oracle.ecc_soft_bwd(img, tau, lam, alpha, U[j], g[..., j, :],
                                 ndim=ndim)["grad_img_absterms"]
        for d in range(ndim):
            sh = [1] * ab.ndim
            sh[ab.ndim - ndim + d] = shape[d]
            t = ab * np.abs(axis_coords(shape[d])).reshape(sh)
            out[j, d] = 4e-6 * np.sqrt(np.sum(t * t))
    return out


def run(img, tau, lam, alpha, U, g, ndim, want_img=True):
    a = np.asarray([alpha], np.float32)
    s, ws = ecc.ecc_soft_ect_fwd(dev(img), dev(tau), lam, dev(a), dev(U), ndim=ndim)
    res = ecc.ecc_soft_ect_bwd(dev(img), dev(tau), lam, dev(a), dev(U), dev(g), ws,
                               want_img=want_img, ndim=ndim)
    return s.cpu().numpy(), {k: v.cpu().numpy() for k, v in res.items()}


def compare(img, tau, lam, alpha, U, g, ndim, want_img=True):
    s, res = run(img, tau, lam, alpha, U, g, ndim, want_img)
    ref_s = oracle.ecc_soft_ect_fwd(img, tau, lam, alpha, U, ndim=ndim)
    ref = oracle.ecc_soft_ect_bwd(img, tau, lam, alpha, U, g, ndim=ndim, want_img=want_img)
    assert s.shape == ref_s.shape
    assert_close(s, ref_s, "S")
    assert_close(res["grad_tau"], ref["grad_tau"], "grad_tau")
    assert_close(res["grad_alpha"][0], ref["grad_alpha"], "grad_alpha")
    assert_close(res["grad_u"], ref["grad_u"], "grad_u",
                 extra=grad_u_allowance(img, tau, lam, alpha, U, g, ndim))
    if want_img:
        assert_close(res["grad_img"], ref["grad_img"], "grad_img",
                     extra=4e-6 * ref["grad_img_absterms"])
    else:
        assert "grad_img" not in res


@pytest.mark.parametrize("shape,batch,ndirs", [((33, 70), 2, 5), ((64, 64), 1, 8), ((5, 7), 3, 3),
                                               ((1, 9), 1, 2), ((9, 10, 33), 2, 3),
                                               ((8, 8, 32), 1, 6)])
def test_ect_parity(shape, batch, ndirs):
    img = synthetic.grf(shape, seed=sum(shape), batch=batch) if min(shape) > 1 else \
        np.random.default_rng(3).random((batch,) + shape).astype(np.float32)
    K = 16
    tau = synthetic.uniform_thresholds(K, -0.4, 1.4)
    U = directions(ndirs, len(shape), seed=ndirs)
    g = synthetic.upstream_grad((batch, ndirs, K), seed=5)
    compare(img, tau, 40.0, 1.0, U, g, len(shape))


@pytest.mark.parametrize("shape,batch,ndirs,K", [((33, 70), 2, 5, 16), ((5, 7), 3, 3, 200),
                                                 ((64, 64), 1, 8, 129), ((9, 10, 33), 2, 3, 16),
                                                 ((8, 8, 32), 1, 6, 300)])
def test_ect_parity_without_the_image_gradient(shape, batch, ndirs, K):
    """The backward the transform takes when no image gradient is wanted runs one block per
    (tile, image, direction) instead of one per (tile, image); threshold counts past one chunk
    of the backward (128) included."""
    img = synthetic.grf(shape, seed=sum(shape) + K, batch=batch)
    tau = synthetic.uniform_thresholds(K, -0.4, 1.4)
    U = directions(ndirs, len(shape), seed=ndirs + K)
    g = synthetic.upstream_grad((batch, ndirs, K), seed=K)
    compare(img, tau, 40.0, 1.0, U, g, len(shape), want_img=False)


@pytest.mark.parametrize("shape,K", [((20, 45), 129), ((6, 9, 40), 300)])
def test_ect_parity_many_thresholds_with_the_image_gradient(shape, K):
    img = synthetic.grf(shape, seed=K, batch=2)
    tau = synthetic.uniform_thresholds(K, -0.4, 1.4)
    U = directions(3, len(shape), seed=K + 1)
    g = synthetic.upstream_grad((2, 3, K), seed=K + 2)
    compare(img, tau, 40.0, 1.0, U, g, len(shape))


def test_one_direction_is_the_soft_ecc_bit_for_bit():
    img = synthetic.grf((50, 70), seed=31, batch=2)
    tau = synthetic.uniform_thresholds(24)
    U = np.asarray([[0.07, -0.11]], np.float32)
    g = synthetic.upstream_grad((2, 1, 24), seed=32)
    a = dev(np.asarray([1.0], np.float32))
    s1, ws1 = ecc.ecc_soft_ect_fwd(dev(img), dev(tau), 50.0, a, dev(U))
    r1 = ecc.ecc_soft_ect_bwd(dev(img), dev(tau), 50.0, a, dev(U), dev(g), ws1, want_img=True)
    s2, ws2 = ecc.ecc_soft_fwd(dev(img), dev(tau), 50.0, a, dev(U[0]))
    r2 = ecc.ecc_soft_bwd(dev(img), dev(tau), 50.0, a, dev(U[0]), dev(g[:, 0]), ws2,
                          want_img=True)
    assert torch.equal(s1[:, 0], s2)
    for k in ("grad_tau", "grad_alpha", "grad_img"):
        assert torch.equal(r1[k], r2[k]), k
    assert torch.equal(r1["grad_u"][0], r2["grad_u"])


def test_ect_autograd_layer():
    img = synthetic.grf((12, 14, 40), seed=33, batch=2)
    tau = dev(synthetic.uniform_thresholds(12)).requires_grad_()
    alpha = torch.ones(1, device=DEV, requires_grad=True)
    U = dev(directions(4, 3, seed=34)).requires_grad_()
    x = dev(img).requires_grad_()
    g = synthetic.upstream_grad((2, 4, 12), seed=35)
    s = ecc.soft_ect(x, tau, alpha, U, 50.0)
    (s * dev(g)).sum().backward()
    ref = oracle.ecc_soft_ect_bwd(img, tau.detach().cpu().numpy(), 50.0, 1.0,
                                  U.detach().cpu().numpy(), g, ndim=3)
    assert_close(tau.grad.cpu().numpy(), ref["grad_tau"], "grad_tau")
    assert_close(alpha.grad.cpu().numpy()[0], ref["grad_alpha"], "grad_alpha")
    assert_close(U.grad.cpu().numpy(), ref["grad_u"], "grad_u",
                 extra=grad_u_allowance(img, tau.detach().cpu().numpy(), 50.0, 1.0,
                                        U.detach().cpu().numpy(), g, 3))
    assert_close(x.grad.cpu().numpy(), ref["grad_img"], "grad_img",
                 extra=4e-6 * ref["grad_img_absterms"])


def test_ect_32_directions_sampled():
    """16 images of 128^2, 32 directions, K = 64: S and every gradient checked on two sampled
    images (upstream gradient zero elsewhere) and all directions."""
    img = synthetic.grf((128, 128), seed=36, batch=16)
    tau = synthetic.uniform_thresholds(64)
    U = directions(32, 2, seed=37)
    g_full = synthetic.upstream_grad((16, 32, 64), seed=38)
    sample = np.asarray([3, 11])
    g = np.zeros_like(g_full)
    g[sample] = g_full[sample]
    s, res = run(img, tau, 50.0, 1.0, U, g, 2)
    ref_s = oracle.ecc_soft_ect_fwd(img[sample], tau, 50.0, 1.0, U, ndim=2)
    ref = oracle.ecc_soft_ect_bwd(img[sample], tau, 50.0, 1.0, U, g[sample], ndim=2)
    assert_close(s[sample], ref_s, "S")
    assert_close(res["grad_tau"], ref["grad_tau"], "grad_tau")
    assert_close(res["grad_alpha"][0], ref["grad_alpha"], "grad_alpha")
    assert_close(res["grad_u"], ref["grad_u"], "grad_u",
                 extra=grad_u_allowance(img[sample], tau, 50.0, 1.0, U, g[sample], 2))
    assert_close(res["grad_img"][sample], ref["grad_img"], "grad_img",
                 extra=4e-6 * ref["grad_img_absterms"])
    others = np.setdiff1d(np.arange(16), sample)
    assert not np.any(res["grad_img"][others])


def test_ect_stats_sum_the_directions():
    img = synthetic.grf((40, 90), seed=39, batch=2)
    tau = synthetic.uniform_thresholds(8)
    U = directions(3, 2, seed=40)
    a = dev(np.asarray([1.0], np.float32))
    _, ws = ecc.ecc_soft_ect_fwd(dev(img), dev(tau), 50.0, a, dev(U))
    st = ecc.ecc_soft_ect_stats(dev(img), 8, 3, ws).cpu().numpy()
    want = 0
    for j in range(3):
        _, wsj = ecc.ecc_soft_fwd(dev(img), dev(tau), 50.0, a, dev(U[j]))
        want += int(ecc.ecc_soft_stats(dev(img), 8, wsj)[0])
    assert st[0] == want
