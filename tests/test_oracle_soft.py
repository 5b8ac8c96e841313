"""Pins for the soft-ECC oracle (CPU only).

The soft ECC replaces the sublevel indicator by a sigmoid (paper notes "Scalable GPU-Accelerated
Euler Characteristic Curves", "Key designs -- differentiable ECC layer (sigmoid relaxation)").
It is pinned by: the lambda -> infinity limit (the hard ECC, itself pinned by homology), fp64
central finite differences for every gradient, the saturation limits S(-inf) = 0 and S(+inf) = 1,
the shift identity sum_p dL/dX_p = -sum_k dL/dtau_k, the alpha/lambda/tau rescaling identity and
the closed form for a pure linear ramp, which fixes the coordinate convention.
"""
import numpy as np
import pytest

import oracle
from euler_characteristic_curves_gb300 import synthetic


def _integer_image(shape, seed, levels=6):
    rng = np.random.default_rng(seed)
    return rng.integers(0, levels, size=shape).astype(np.float32)


@pytest.mark.parametrize("shape", [(7, 9), (2, 5, 6), (1, 8), (4, 4, 1)])
def test_large_lambda_recovers_hard_ecc(shape):
    img = _integer_image(shape, 1)
    # thresholds at half-integers -0.5 .. 5.5; |u . x| < 0.2 never crosses a half-integer
    tau = (np.arange(7) - 0.5).astype(np.float32)
    u = np.full(len(shape), 0.09, np.float32)
    s = oracle.ecc_soft_fwd(img, tau, 1.0e4, 1.0, u)
    hard = oracle.ecc_hard(img, 7, -0.5, 5.5)
    np.testing.assert_allclose(s, hard.astype(np.float64), rtol=0, atol=1e-12)


def test_saturation_limits():
    f = synthetic.grf((12, 15), 3)
    tau = np.asarray([-1000.0, 1000.0], np.float32)
    s = oracle.ecc_soft_fwd(f, tau, 50.0, 1.0, [0.05, -0.03])
    assert abs(s[0]) < 1e-300 and abs(s[1] - 1.0) < 1e-12
    f3 = synthetic.grf((5, 6, 7), 4)
    s = oracle.ecc_soft_fwd(f3, tau, 50.0, 1.0, [0.05, -0.03, 0.02])
    assert abs(s[0]) < 1e-300 and abs(s[1] - 1.0) < 1e-12


@pytest.mark.parametrize("axis", [0, 1])
@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_linear_ramp_closed_form(axis, sign):
    """f = 0, u along one axis: every sublevel set is a box, and only the first slab to enter
    changes chi. For u_a > 0 that slab sits at coordinate -1, so S(t) = sigma(lam (t + u_a)); for
    u_a < 0 it sits at +1 and S(t) = sigma(lam (t - u_a))."""
    shape = (6, 9)
    f = np.zeros(shape, np.float32)
    u = np.zeros(2, np.float32)
    u[axis] = np.float32(0.3 * sign)
    tau = np.linspace(-0.6, 0.6, 13).astype(np.float32)
    lam = 7.0
    s = oracle.ecc_soft_fwd(f, tau, lam, 1.0, u)
    ua = float(u[axis])
    edge = -ua if ua > 0 else ua  # X of the first slab: u_a * (-1) or u_a * (+1)
    expect = 1.0 / (1.0 + np.exp(-lam * (tau.astype(np.float64) - edge)))
    np.testing.assert_allclose(s, expect, rtol=1e-13, atol=1e-15)
    # and its gradient with respect to u_a: dS/du_a = lam s (1 - s) * (+1 for u_a > 0, -1 else)
    g = np.linspace(-1, 1, 13)
    res = oracle.ecc_soft_bwd(f, tau, lam, 1.0, u, g)
    d = lam * expect * (1 - expect) * (1.0 if ua > 0 else -1.0)
    np.testing.assert_allclose(res["grad_u"][axis], np.sum(g * d), rtol=1e-12)
    # (the other component is a subgradient: X ties along that axis, so it is not checked)


@pytest.mark.parametrize("shape,u,pixel", [((3, 4), (0.0, 0.0), (0, 0)),
                                           ((5, 7), (0.0, 0.0), (0, 0)),
                                           ((3, 5), (0.0, 0.3), (0, 0)),
                                           ((3, 5), (0.0, -0.3), (0, 4)),
                                           ((4, 3), (-0.3, 0.0), (3, 0)),
                                           ((4, 6), (-0.2, -0.1), (3, 5)),
                                           ((3, 4, 5), (0.0, 0.0, 0.0), (0, 0, 0)),
                                           ((3, 4, 5), (-0.3, 0.0, 0.0), (2, 0, 0)),
                                           ((3, 4, 5), (0.0, -0.3, 0.0), (0, 3, 0)),
                                           ((3, 4, 5), (0.0, 0.0, -0.2), (0, 0, 4)),
                                           ((3, 4, 5), (0.1, -0.2, -0.3), (0, 3, 4))])
def test_gradient_lands_on_the_first_entering_pixel(shape, u, pixel):
    """f = 0, X = u . x (constant when u = 0). Every sublevel set is a box, so only the first
    pixel to enter has a non-zero local contribution (+1), and the image gradient sits on that
    pixel alone: the first pixel in index order when values tie ("lower index enters first"),
    otherwise the corner where X is smallest -- which corner pins the axis order of u and x."""
    f = np.zeros(shape, np.float32)
    lam, tau = 4.0, np.asarray([0.1], np.float32)
    r = oracle.ecc_soft_bwd(f, tau, lam, 1.0, np.asarray(u, np.float32), np.ones(1))
    gi = r["grad_img"]
    nz = np.argwhere(gi != 0)
    assert [tuple(x) for x in nz] == [pixel]
    # X of that corner: each axis adds -|u_d| (coordinate -1 for u_d > 0, +1 for u_d < 0)
    x = sum(-float(np.float32(abs(ud))) for ud in u)
    s = 1.0 / (1.0 + np.exp(-lam * (0.1 - x)))
    # dL/dX = -lambda s (1 - s) for the only contributing vertex, grad_img = alpha dL/dX
    assert abs(gi[pixel] + lam * s * (1 - s)) < 1e-7


def test_alpha_rescaling_identity():
    """With u = 0, S(f; alpha, lam, tau) = S(f; 1, lam * alpha, tau / alpha)."""
    f = synthetic.grf((10, 11), 5)
    tau = np.linspace(0, 1, 9).astype(np.float32)
    a = 2.0  # exact in fp32, so tau / alpha is exact too
    s1 = oracle.ecc_soft_fwd(f, tau, 6.0, a, [0.0, 0.0])
    s2 = oracle.ecc_soft_fwd(f, (tau / a).astype(np.float32), 12.0, 1.0, [0.0, 0.0])
    np.testing.assert_allclose(s1, s2, rtol=1e-12, atol=1e-14)


def _fd_check(shape, seed, lam, K):
    rng = np.random.default_rng(seed)
    # generic values: distinct enough that a perturbation of h never reorders neighbours
    f = rng.permutation(np.prod(shape)).reshape(shape).astype(np.float32) / np.prod(shape)
    tau = np.linspace(0.05, 0.95, K).astype(np.float32)
    alpha = 1.25
    u = (0.05 * (np.arange(len(shape)) + 1)).astype(np.float32)
    g = rng.standard_normal(K)

    # the oracle takes fp32 inputs, so every perturbation is a power-of-two step that fp32
    # represents exactly; the difference quotient divides by the realised (exact) step.
    def L(f_=f, tau_=tau, alpha_=alpha, u_=u):
        return float(np.sum(g * oracle.ecc_soft_fwd(f_, tau_, lam, alpha_, u_)))

    res = oracle.ecc_soft_bwd(f, tau, lam, alpha, u, g)
    step = np.float32(2.0 ** -12)

    for k in range(K):
        tp, tm = tau.copy(), tau.copy()
        tp[k] += step
        tm[k] -= step
        fd = (L(tau_=tp) - L(tau_=tm)) / (float(tp[k]) - float(tm[k]))
        assert abs(fd - res["grad_tau"][k]) <= 1e-5 * max(1.0, abs(fd)), (k, fd, res["grad_tau"][k])
    ap, am = np.float32(alpha + step), np.float32(alpha - step)
    fd = (L(alpha_=ap) - L(alpha_=am)) / (float(ap) - float(am))
    assert abs(fd - res["grad_alpha"]) <= 1e-5 * max(1.0, abs(fd))
    for d in range(len(shape)):
        up, um = u.copy(), u.copy()
        up[d] += step
        um[d] -= step
        fd = (L(u_=up) - L(u_=um)) / (float(up[d]) - float(um[d]))
        assert abs(fd - res["grad_u"][d]) <= 1e-5 * max(1.0, abs(fd))
    flat = f.reshape(-1)
    for p in rng.choice(flat.size, size=min(12, flat.size), replace=False):
        fp, fm = flat.copy(), flat.copy()
        fp[p] += np.float32(2.0 ** -16)
        fm[p] -= np.float32(2.0 ** -16)
        fd = (L(f_=fp.reshape(shape)) - L(f_=fm.reshape(shape))) / (float(fp[p]) - float(fm[p]))
        got = res["grad_img"].reshape(-1)[p]
        assert abs(fd - got) <= 1e-5 * max(1.0, abs(fd)), (p, fd, got)


@pytest.mark.parametrize("shape,seed", [((5, 6), 0), ((3, 4, 5), 1), ((1, 7), 2), ((6, 1), 3)])
def test_gradients_match_finite_differences(shape, seed):
    _fd_check(shape, seed, lam=3.0, K=5)


def test_shift_identity_and_batch_sum():
    f = synthetic.grf((9, 13), 8, batch=3)
    tau = np.linspace(0, 1, 17).astype(np.float32)
    g = synthetic.upstream_grad((3, 17), 9)
    alpha = 1.5
    res = oracle.ecc_soft_bwd(f, tau, 20.0, alpha, [0.1, -0.2], g, ndim=2)
    lhs = np.sum(res["grad_img"]) / alpha
    assert abs(lhs + np.sum(res["grad_tau"])) <= 1e-9 * max(1.0, np.abs(res["grad_tau"]).sum())
    # parameters are shared across the batch: batch gradients are sums of per-image gradients
    parts = [oracle.ecc_soft_bwd(f[b], tau, 20.0, alpha, [0.1, -0.2], g[b]) for b in range(3)]
    np.testing.assert_allclose(res["grad_tau"], sum(p["grad_tau"] for p in parts), rtol=1e-12,
                               atol=1e-9)
    np.testing.assert_allclose(res["grad_alpha"], sum(p["grad_alpha"] for p in parts),
                               rtol=1e-12)
    s = oracle.ecc_soft_fwd(f, tau, 20.0, alpha, [0.1, -0.2], ndim=2)
    for b in range(3):
        np.testing.assert_array_equal(s[b], oracle.ecc_soft_fwd(f[b], tau, 20.0, alpha,
                                                                [0.1, -0.2]))


def test_u_zero_alpha_one_is_soft_ecc_of_f():
    """alpha = 1, u = 0: the filtration is f itself, so large lambda gives the hard ECC of f."""
    f = synthetic.quantise_u8(synthetic.grf((14, 10), 10)).astype(np.float32)
    tau = (np.arange(0, 256, 15) + 0.5).astype(np.float32)
    s = oracle.ecc_soft_fwd(f, tau, 1.0e4, 1.0, [0.0, 0.0])
    hard = oracle.ecc_hard(f, 256, 0.0, 255.0)[np.arange(0, 256, 15)]
    np.testing.assert_allclose(s, hard.astype(np.float64), atol=1e-12)


# ---------------------------------------------------------------------------------------------
# Soft Euler characteristic transform (several directions)
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("shape", [(4, 5), (3, 4, 5)])
def test_ect_closed_form_on_a_flat_image(shape):
    """f = 0: along every direction u_j each sublevel set of X_j = u_j . x is a staircase region
    of the grid, contractible whenever non-empty, so only the first voxel to enter contributes
    and S_j(t) = sigma(lam (t - X_min,j)), X_min,j = -sum_d |u_jd| (a corner of the grid). The
    u-gradient of each direction follows from dX_min,j / du_jd = -sign(u_jd)."""
    f = np.zeros(shape, np.float32)
    rng = np.random.default_rng(len(shape))
    U = rng.normal(0, 0.3, size=(5, len(shape))).astype(np.float32)
    U[1, 0] = 0.0  # one direction with a tie along an axis
    tau = np.linspace(-1.0, 1.0, 7).astype(np.float32)
    lam = 5.0
    s = oracle.ecc_soft_ect_fwd(f, tau, lam, 1.0, U)
    assert s.shape == (5, 7)
    g = rng.standard_normal((5, 7))
    res = oracle.ecc_soft_ect_bwd(f, tau, lam, 1.0, U, g)
    for j in range(5):
        xmin = -sum(abs(float(x)) for x in U[j])
        want = 1.0 / (1.0 + np.exp(-lam * (tau.astype(np.float64) - xmin)))
        np.testing.assert_allclose(s[j], want, rtol=1e-12, atol=1e-15)
        dsdx = -lam * want * (1 - want)  # dS/dX_min
        for d in range(len(shape)):
            if U[j, d] != 0.0:
                want_gu = np.sum(g[j] * dsdx) * (-np.sign(U[j, d]))
                np.testing.assert_allclose(res["grad_u"][j, d], want_gu, rtol=1e-10)


def test_ect_of_one_direction_is_the_soft_ecc_and_batches_stack():
    img = synthetic.grf((9, 11), 21, batch=3)
    tau = synthetic.uniform_thresholds(6)
    U = np.asarray([[0.1, -0.2], [0.0, 0.0], [-0.3, 0.05]], np.float32)
    s = oracle.ecc_soft_ect_fwd(img, tau, 40.0, 1.0, U, ndim=2)
    assert s.shape == (3, 3, 6)
    for j in range(3):
        np.testing.assert_array_equal(s[:, j], oracle.ecc_soft_fwd(img, tau, 40.0, 1.0, U[j], ndim=2))


@pytest.mark.parametrize("shape", [(5, 6), (3, 4, 5)])
def test_ect_gradients_match_finite_differences(shape):
    """The transform's backward against central differences of its own forward, with two images
    and three directions: catches a direction's upstream slice or its u-gradient row taken from
    the wrong place (the single-direction pins cannot)."""
    rng = np.random.default_rng(7)
    n = int(np.prod(shape))
    f = np.stack([rng.permutation(n).reshape(shape) for _ in range(2)]).astype(np.float32) / n
    K, nd, lam, alpha = 4, 3, 3.0, 1.25
    tau = np.linspace(0.1, 0.9, K).astype(np.float32)
    U = (0.05 * rng.standard_normal((nd, len(shape)))).astype(np.float32)
    g = rng.standard_normal((2, nd, K))

    def L(f_=f, tau_=tau, alpha_=alpha, U_=U):
        s = oracle.ecc_soft_ect_fwd(f_, tau_, lam, alpha_, U_, ndim=len(shape))
        assert s.shape == g.shape
        return float(np.sum(g * s))

    res = oracle.ecc_soft_ect_bwd(f, tau, lam, alpha, U, g, ndim=len(shape))
    step = np.float32(2.0 ** -12)

    def close(fd, got):
        return abs(fd - got) <= 1e-5 * max(1.0, abs(fd))

    for k in range(K):
        tp, tm = tau.copy(), tau.copy()
        tp[k] += step
        tm[k] -= step
        fd = (L(tau_=tp) - L(tau_=tm)) / (float(tp[k]) - float(tm[k]))
        assert close(fd, res["grad_tau"][k]), (k, fd, res["grad_tau"][k])
    ap, am = np.float32(alpha + step), np.float32(alpha - step)
    assert close((L(alpha_=ap) - L(alpha_=am)) / (float(ap) - float(am)), res["grad_alpha"])
    for j in range(nd):
        for d in range(len(shape)):
            Up, Um = U.copy(), U.copy()
            Up[j, d] += step
            Um[j, d] -= step
            fd = (L(U_=Up) - L(U_=Um)) / (float(Up[j, d]) - float(Um[j, d]))
            assert close(fd, res["grad_u"][j, d]), (j, d, fd, res["grad_u"][j, d])
    flat = f.reshape(-1)
    for p in rng.choice(flat.size, size=10, replace=False):
        fp, fm = flat.copy(), flat.copy()
        fp[p] += np.float32(2.0 ** -16)
        fm[p] -= np.float32(2.0 ** -16)
        fd = (L(f_=fp.reshape(f.shape)) - L(f_=fm.reshape(f.shape))) / (float(fp[p]) - float(fm[p]))
        got = res["grad_img"].reshape(-1)[p]
        assert close(fd, got), (p, fd, got)


def test_pool_of_images_equals_the_batch():
    """The per-image pool helper gives the batch oracle's S and gradients."""
    from tests import _oracle_pool

    f = synthetic.grf((11, 15), 41, batch=3)
    tau = np.linspace(0, 1, 9).astype(np.float32)
    g = synthetic.upstream_grad((3, 9), 42)
    u = np.asarray([0.1, -0.2], np.float32)
    s, r = _oracle_pool.soft_batch(f, tau, 20.0, 1.0, u, g, ndim=2)
    np.testing.assert_array_equal(s, oracle.ecc_soft_fwd(f, tau, 20.0, 1.0, u, ndim=2))
    ref = oracle.ecc_soft_bwd(f, tau, 20.0, 1.0, u, g, ndim=2)
    np.testing.assert_allclose(r["grad_tau"], ref["grad_tau"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r["grad_alpha"], ref["grad_alpha"], rtol=1e-12)
    np.testing.assert_allclose(r["grad_u"], ref["grad_u"], rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(r["grad_img"], ref["grad_img"])


def test_grad_tau_absterms_bounds_and_single_vertex_closed_form():
    """grad_tau_absterms (the scale of the cancellation in grad_tau) against what fixes it: for a
    1 x 1 image the only cell is its vertex (sign +1), so every term of grad_tau[k] is
    g_k lambda s (1 - s) with s = sigma(lambda (t_k - alpha f)) and the sum of |terms| is the
    same closed form with |g_k|; for any image it bounds |grad_tau| (triangle inequality) and
    equals it where every term has one sign (g >= 0 on a 1 x 1 image)."""
    lam, alpha, f = 30.0, 1.0, 0.4
    tau = np.linspace(0.0, 1.0, 9).astype(np.float32)
    g = np.asarray([[0.5, -1.0, 2.0, -0.25, 1.0, -3.0, 0.75, 0.1, -0.6]])
    img = np.full((1, 1, 1), f, np.float32)
    r = oracle.ecc_soft_bwd(img, tau, lam, alpha, np.zeros(2, np.float32), g, ndim=2,
                            want_img=False)
    s = 1.0 / (1.0 + np.exp(-lam * (tau.astype(np.float64) - np.float32(f))))
    w = lam * s * (1.0 - s)
    np.testing.assert_allclose(r["grad_tau"], g[0] * w, rtol=1e-12, atol=0)
    np.testing.assert_allclose(r["grad_tau_absterms"], np.abs(g[0]) * w, rtol=1e-12, atol=0)
    rp = oracle.ecc_soft_bwd(img, tau, lam, alpha, np.zeros(2, np.float32), np.abs(g), ndim=2,
                             want_img=False)
    np.testing.assert_array_equal(rp["grad_tau_absterms"], rp["grad_tau"])
    img = synthetic.grf((7, 9), 61, batch=2)
    tau = synthetic.uniform_thresholds(20)
    g = synthetic.upstream_grad((2, 20), seed=62)
    r = oracle.ecc_soft_bwd(img, tau, 40.0, 1.0, np.asarray([0.1, -0.05], np.float32), g,
                            ndim=2, want_img=False)
    assert np.all(np.abs(r["grad_tau"]) <= r["grad_tau_absterms"] * (1 + 1e-12))
    assert np.all(r["grad_tau_absterms"] > 0)
