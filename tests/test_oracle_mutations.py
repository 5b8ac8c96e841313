"""The pins catch plausible mistakes: each test plants one mistake in a copy of the oracle's C
source (on the CPU), builds it, swaps it in, and checks that the pins that should notice do.

Mistakes planted: a flipped sign for odd-dimensional cells, a dropped cell type, '<' for '<=' in
the threshold comparison, a transposed offset for one axis, a reversed sigmoid argument, a wrong
sign in the backward pass, the opposite tie rule for the cell owner, and swapped coordinate axes;
and, in a copy of the transform's Python bookkeeping, a direction reading another direction's
upstream gradient or writing its u-gradient to another row.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle
from euler_characteristic_curves_gb300 import synthetic
from tests import _topology as topo

SRC = os.path.join(os.path.dirname(oracle.__file__), "ecc_oracle.c")


def _build_mutant(tmp_path, old, new):
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation anchor not found: {old!r}"
    text = text.replace(old, new)
    src = tmp_path / "mutant.c"
    src.write_text(text)
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off", str(src),
                    "-o", str(lib), "-lm"], check=True)
    return str(lib)


@pytest.fixture
def swap_oracle(monkeypatch):
    import ctypes

    def use(path):
        oracle._load()  # make sure the real library's argtypes exist, then mirror them
        lib = ctypes.CDLL(path)
        for name in ("oracle_thresholds", "oracle_ecc_hard", "oracle_ecc_soft_fwd",
                     "oracle_ecc_soft_bwd"):
            getattr(lib, name).argtypes = getattr(oracle._lib, name).argtypes
            getattr(lib, name).restype = getattr(oracle._lib, name).restype
        monkeypatch.setattr(oracle, "_lib", lib)

    return use


def gradient_lands_on(shape, u, pixel):
    """f = 0 (X = u . x): the whole image gradient sits on one pixel."""
    f = np.zeros(shape, np.float32)
    r = oracle.ecc_soft_bwd(f, np.asarray([0.1], np.float32), 4.0, 1.0, u, np.ones(1))
    gi = r["grad_img"]
    nz = np.argwhere(gi != 0)
    return len(nz) == 1 and tuple(nz[0]) == pixel


def hard_pins_pass():
    """A compact set of the hard-ECC pins; True when all hold."""
    # exhaustive 3x3 binary grids against flood fill
    codes = np.arange(1 << 9)
    masks = ((codes[:, None] >> np.arange(9)) & 1).astype(bool).reshape(-1, 3, 3)
    ecc = oracle.ecc_hard(np.where(masks, 0, 1).astype(np.uint8), 2, 0.0, 1.0, ndim=2)
    if not np.array_equal(ecc[:, 0], [topo.chi_2d_flood(m) for m in masks]):
        return False
    # 3-D: every 2x2x2 grid against homology + flood fill
    for code in range(256):
        m = ((code >> np.arange(8)) & 1).astype(bool).reshape(2, 2, 2)
        b = topo.betti(m)
        chi = topo.b0(m) - b[1] + topo.cavities(m)
        if oracle.ecc_hard(np.where(m, 0, 1).astype(np.uint8), 2, 0.0, 1.0)[0] != chi:
            return False
    # integer thresholds: a value equal to a threshold enters at it
    if oracle.ecc_hard(np.full((3, 3), 2, np.uint8), 4, 0.0, 3.0).tolist() != [0, 0, 1, 1]:
        return False
    # symmetry under transposition of a rectangular 3-D field
    f = synthetic.grf((4, 5, 6), 1)
    if not np.array_equal(oracle.ecc_hard(f, 16, 0.0, 1.0),
                          oracle.ecc_hard(np.ascontiguousarray(f.transpose(2, 1, 0)), 16, 0.0,
                                          1.0)):
        return False
    return True


def soft_pins_pass():
    """A compact set of the soft-ECC pins; True when all hold."""
    img = np.random.default_rng(1).integers(0, 6, size=(6, 7)).astype(np.float32)
    tau = (np.arange(7) - 0.5).astype(np.float32)
    s = oracle.ecc_soft_fwd(img, tau, 1.0e4, 1.0, [0.09, 0.09])
    if not np.allclose(s, oracle.ecc_hard(img, 7, -0.5, 5.5), atol=1e-12):
        return False
    # linear-ramp closed form along axis 1 (fixes the coordinate convention)
    f = np.zeros((5, 8), np.float32)
    t = np.linspace(-0.5, 0.5, 9).astype(np.float32)
    s = oracle.ecc_soft_fwd(f, t, 7.0, 1.0, [0.0, 0.3])
    want = 1.0 / (1.0 + np.exp(-7.0 * (t.astype(np.float64) + np.float64(np.float32(0.3)))))
    if not np.allclose(s, want, rtol=1e-12):
        return False
    # finite differences for the gradients, on distinct values
    rng = np.random.default_rng(2)
    f = (rng.permutation(30).reshape(5, 6) / 30.0).astype(np.float32)
    tau = np.linspace(0.1, 0.9, 4).astype(np.float32)
    g = rng.standard_normal(4)
    u = np.asarray([0.05, 0.1], np.float32)
    res = oracle.ecc_soft_bwd(f, tau, 3.0, 1.25, u, g)
    step = np.float32(2.0 ** -12)
    for k in range(4):
        tp, tm = tau.copy(), tau.copy()
        tp[k] += step
        tm[k] -= step
        fd = (np.sum(g * oracle.ecc_soft_fwd(f, tp, 3.0, 1.25, u)) -
              np.sum(g * oracle.ecc_soft_fwd(f, tm, 3.0, 1.25, u))) / (float(tp[k]) - float(tm[k]))
        if abs(fd - res["grad_tau"][k]) > 1e-5 * max(1.0, abs(fd)):
            return False
    flat = f.reshape(-1)
    for p in (3, 17, 25):
        fp, fm = flat.copy(), flat.copy()
        fp[p] += np.float32(2.0 ** -16)
        fm[p] -= np.float32(2.0 ** -16)
        fd = (np.sum(g * oracle.ecc_soft_fwd(fp.reshape(5, 6), tau, 3.0, 1.25, u)) -
              np.sum(g * oracle.ecc_soft_fwd(fm.reshape(5, 6), tau, 3.0, 1.25, u))) / (
                  float(fp[p]) - float(fm[p]))
        if abs(fd - res["grad_img"].reshape(-1)[p]) > 1e-5 * max(1.0, abs(fd)):
            return False
    # ties and axis convention through where the gradient lands (see test_oracle_soft.py)
    if not gradient_lands_on((3, 4), [0.0, 0.0], (0, 0)):
        return False
    if not gradient_lands_on((3, 5), [0.0, -0.3], (0, 4)):
        return False
    if not gradient_lands_on((4, 3), [-0.3, 0.0], (3, 0)):
        return False
    return True


def test_unmutated_oracle_passes_the_pin_subsets():
    assert hard_pins_pass()
    assert soft_pins_pass()


HARD_MUTANTS = [
    ("flipped sign of odd cells", "(popcount_small(S) & 1) ? -1 : 1",
     "(popcount_small(S) & 1) ? 1 : -1"),
    ("squares dropped", "        if (!cell_exists(&g, idx, S)) continue;\n                int k = 0;",
     "        if (!cell_exists(&g, idx, S) || S == 3) continue;\n                int k = 0;"),
    ("strict threshold comparison", "if (v <= tau[mid])", "if (v < tau[mid])"),
    ("one axis offset transposed", "if (T >> d & 1) off += g->stride[d];",
     "if (T >> d & 1) off += g->stride[g->ndim - 1 - d];"),
]

SOFT_MUTANTS = [
    ("reversed sigmoid argument", "sigmoid(lambda * ((double)tau[k] - xmax))",
     "sigmoid(lambda * (xmax - (double)tau[k]))"),
    ("backward sign", "dX[owner] -= term;", "dX[owner] += term;"),
    ("opposite tie rule", "(X[q] == X[best] && q > best)", "(X[q] == X[best] && q < best)"),
    ("swapped coordinate axes", "x = x + u[d] * axis_coord(idx[d], g->n[d]);",
     "x = x + u[g->ndim - 1 - d] * axis_coord(idx[d], g->n[d]);"),
]


@pytest.mark.parametrize("name,old,new", HARD_MUTANTS)
def test_hard_pins_catch(tmp_path, swap_oracle, name, old, new):
    swap_oracle(_build_mutant(tmp_path, old, new))
    assert not hard_pins_pass(), f"mutation not caught: {name}"


@pytest.mark.parametrize("name,old,new", SOFT_MUTANTS)
def test_soft_pins_catch(tmp_path, swap_oracle, name, old, new):
    swap_oracle(_build_mutant(tmp_path, old, new))
    assert not soft_pins_pass(), f"mutation not caught: {name}"


def _mutant_python(monkeypatch, func_name, old, new):
    """Plant a mistake in a copy of one of the oracle's Python functions and swap it in."""
    import inspect
    import textwrap

    src = textwrap.dedent(inspect.getsource(getattr(oracle, func_name)))
    assert src.count(old) == 1, f"mutation anchor not found: {old!r}"
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), f"<mutant {func_name}>", "exec"), ns)
    monkeypatch.setattr(oracle, func_name, ns[func_name])


@pytest.mark.parametrize("old,new", [
    ("go[..., j, :]", "go[..., (j + 1) % U.shape[0], :]"),       # another direction's upstream
    ('res["grad_u"][j] = ', 'res["grad_u"][(j + 1) % U.shape[0]] = '),  # u-gradient row swapped
])
def test_transform_pin_catches_direction_bookkeeping(monkeypatch, old, new):
    from tests import test_oracle_soft as pins

    pins.test_ect_gradients_match_finite_differences((5, 6))  # the real oracle passes
    _mutant_python(monkeypatch, "ecc_soft_ect_bwd", old, new)
    with pytest.raises(AssertionError):
        pins.test_ect_gradients_match_finite_differences((5, 6))
