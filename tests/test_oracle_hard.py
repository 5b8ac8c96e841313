"""Pins for the hard-ECC oracle (CPU only).

Each test checks the oracle against something other than itself: flood-fill Betti numbers,
GF(2) homology, closed forms, and invariants of the Euler characteristic (symmetry, additivity
over disjoint unions, inclusion-exclusion over overlapping slabs, monotone relabelling).
"""
import itertools
import os

import numpy as np
import pytest

import oracle
from euler_characteristic_curves_gb300 import synthetic
from tests import _topology as topo

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_curves.txt")


def chi_of_mask(mask):
    """ECC of a binary mask through the oracle: foreground = value 0, background = value 1,
    thresholds {0, 1}; entry 0 is the Euler characteristic of the foreground."""
    img = np.where(mask, 0, 1).astype(np.uint8)
    return int(oracle.ecc_hard(img, 2, 0.0, 1.0)[0])


# ----------------------------------------------------------------------------- thresholds

def test_thresholds_formula():
    t = oracle.thresholds(5, -1.0, 3.0)
    assert t.tolist() == [-1.0, 0.0, 1.0, 2.0, 3.0]
    assert oracle.thresholds(1, 0.25, 0.75).tolist() == [0.75]
    t = oracle.thresholds(256, 0.0, 255.0)
    assert t.tolist() == [float(k) for k in range(256)]
    t = oracle.thresholds(1024, 0.0, 1.0)
    assert t[0] == 0.0 and t[-1] == 1.0
    assert np.all(np.diff(t) > 0)
    np.testing.assert_allclose(t, np.arange(1024) / 1023.0, rtol=0, atol=1e-15)


# ----------------------------------------------------------------------------- brute force 2-D

@pytest.mark.parametrize("shape", [(1, 1), (1, 5), (4, 1), (2, 2), (2, 3), (3, 3), (3, 4), (4, 4)])
def test_exhaustive_binary_2d_matches_flood_fill(shape):
    """Every binary grid of the shape: oracle chi == b0 (4-conn) - holes (8-conn complement)."""
    n = shape[0] * shape[1]
    codes = np.arange(1 << n, dtype=np.int64)
    masks = ((codes[:, None] >> np.arange(n)) & 1).astype(bool).reshape((-1,) + shape)
    imgs = np.where(masks, 0, 1).astype(np.uint8)
    ecc = oracle.ecc_hard(imgs, 2, 0.0, 1.0, ndim=2)
    assert np.all(ecc[:, 1] == 1)  # the whole grid is contractible
    expect = np.array([topo.chi_2d_flood(m) for m in masks])
    np.testing.assert_array_equal(ecc[:, 0], expect)


def test_homology_helper_agrees_with_flood_fill():
    rng = np.random.default_rng(0)
    for _ in range(60):
        m = rng.random((3, 3, 3)) < 0.6
        b = topo.betti(m)
        assert b[0] == topo.b0(m)
        assert b[2] == topo.cavities(m)


# ----------------------------------------------------------------------------- brute force 3-D

def _check_3d_mask(m):
    b = topo.betti(m)
    chi = topo.b0(m) - b[1] + topo.cavities(m)
    assert chi_of_mask(m) == chi, (m.astype(int), b)


def test_exhaustive_binary_2x2x2():
    for code in range(256):
        m = ((code >> np.arange(8)) & 1).astype(bool).reshape(2, 2, 2)
        _check_3d_mask(m)


@pytest.mark.parametrize("shape,density,count", [((3, 3, 3), 0.5, 150), ((3, 3, 3), 0.75, 150),
                                                 ((4, 4, 4), 0.6, 60), ((2, 3, 5), 0.5, 100)])
def test_random_binary_3d_matches_homology(shape, density, count):
    rng = np.random.default_rng(hash(shape) % 1000 + int(density * 100))
    for _ in range(count):
        _check_3d_mask(rng.random(shape) < density)


# ----------------------------------------------------------------------------- closed forms

def test_single_pixel_and_boxes():
    for shape in [(1, 1), (7, 1), (1, 9), (5, 6), (1, 1, 1), (3, 4, 5)]:
        img = np.zeros(shape, np.float32)
        assert oracle.ecc_hard(img, 3, -1.0, 1.0).tolist() == [0, 1, 1]
    img = np.full((6, 7), 2.0, np.float32)
    img[3, 4] = 0.0  # one pixel below the others
    assert oracle.ecc_hard(img, 3, 0.0, 2.0).tolist() == [1, 1, 1]


def test_constant_image_is_a_step():
    img = np.full((5, 8), 0.5, np.float32)
    out = oracle.ecc_hard(img, 11, 0.0, 1.0)
    assert out.tolist() == [0] * 5 + [1] * 6


def test_annulus_and_k_blobs_2d():
    a = np.ones((9, 9), np.float32)
    a[2:7, 2:7] = 0.0
    a[4, 4] = 1.0  # a ring of zeros around a high centre
    assert oracle.ecc_hard(a, 2, 0.0, 1.0).tolist() == [0, 1]
    rng = np.random.default_rng(3)
    for k in range(1, 9):
        img = np.ones((20, 40), np.float32)
        for j in range(k):  # separated 2x3 blobs
            img[2 + (j % 2) * 8: 5 + (j % 2) * 8, 2 + j * 4: 4 + j * 4] = rng.random() * 0.5
        out = oracle.ecc_hard(img, 2, 0.5, 1.0)
        assert out.tolist() == [k, 1]


def test_shell_and_torus_3d():
    shell = np.zeros((5, 5, 5), np.float32)
    shell[1:4, 1:4, 1:4] = 1.0
    shell[2, 2, 2] = 2.0  # the inner cube's centre stays out: the sublevel set is a hollow shell
    shell = np.pad(np.ones((3, 3, 3), np.float32) * 2.0, 1, constant_values=3.0)
    shell[1:4, 1:4, 1:4] = 1.0
    shell[2, 2, 2] = 2.0
    assert oracle.ecc_hard(shell, 3, 1.0, 3.0).tolist() == [2, 1, 1]
    torus = np.ones((3, 6, 6), np.float32)
    torus[1, 1:5, 1:5] = 0.0
    torus[1, 2:4, 2:4] = 1.0  # a square ring in the middle plane: a solid torus
    assert oracle.ecc_hard(torus, 2, 0.0, 1.0).tolist() == [0, 1]


def _parse_golden():
    cases = []
    with open(GOLDEN) as fh:
        block = []
        for line in fh:
            line = line.split("#", 1)[0].rstrip()
            if not line:
                continue
            if line.startswith("case"):
                if block:
                    cases.append(block)
                block = [line]
            else:
                block.append(line)
        if block:
            cases.append(block)
    parsed = []
    for blk in cases:
        head = dict(kv.split("=") for kv in blk[0].split()[1:])
        rows = [list(map(float, r.split())) for r in blk[1:-1]]
        expect = list(map(int, blk[-1].split("=")[1].split()))
        shape = tuple(int(s) for s in head["shape"].split("x"))
        img = np.asarray(rows, np.float32).reshape(shape)
        parsed.append((head["name"], img, int(head["nbins"]), float(head["vmin"]),
                       float(head["vmax"]), expect))
    return parsed


def test_hand_derived_curves():
    cases = _parse_golden()
    assert len(cases) >= 5
    for name, img, nbins, vmin, vmax, expect in cases:
        got = oracle.ecc_hard(img, nbins, vmin, vmax).tolist()
        assert got == expect, name
        if np.all(img == np.round(img)) and img.min() >= 0 and img.max() <= 255:
            assert oracle.ecc_hard(img.astype(np.uint8), nbins, vmin, vmax).tolist() == expect


# ----------------------------------------------------------------------------- invariants

def _rand_field(shape, seed):
    return synthetic.grf(shape, seed)


@pytest.mark.parametrize("shape", [(17, 23), (32, 32)])
def test_symmetries_2d(shape):
    f = _rand_field(shape, 11)
    ref = oracle.ecc_hard(f, 64, 0.0, 1.0)
    for k in range(4):
        for flip in (False, True):
            g = np.rot90(f, k)
            g = g[:, ::-1] if flip else g
            np.testing.assert_array_equal(oracle.ecc_hard(np.ascontiguousarray(g), 64, 0.0, 1.0),
                                          ref)


def test_symmetries_3d():
    f = _rand_field((6, 7, 8), 12)
    ref = oracle.ecc_hard(f, 32, 0.0, 1.0)
    for perm in itertools.permutations(range(3)):
        for flips in itertools.product((False, True), repeat=3):
            g = np.transpose(f, perm)
            sl = tuple(slice(None, None, -1) if fl else slice(None) for fl in flips)
            np.testing.assert_array_equal(
                oracle.ecc_hard(np.ascontiguousarray(g[sl]), 32, 0.0, 1.0), ref)


def test_extreme_thresholds():
    f = _rand_field((40, 30), 13)
    out = oracle.ecc_hard(f, 16, float(f.min()) - 1.0, float(f.max()))
    assert out[0] == 0 and out[-1] == 1
    out = oracle.ecc_hard(f, 8, -3.0, -2.0)
    assert out.tolist() == [0] * 8


def test_disjoint_union_additivity():
    a = _rand_field((20, 30), 14)
    b = _rand_field((25, 30), 15)
    sep = np.full((1, 30), 5.0, np.float32)  # above vmax: never enters, separates the halves
    joined = np.concatenate([a, sep, b], axis=0)
    ea = oracle.ecc_hard(a, 50, 0.0, 1.0)
    eb = oracle.ecc_hard(b, 50, 0.0, 1.0)
    np.testing.assert_array_equal(oracle.ecc_hard(joined, 50, 0.0, 1.0), ea + eb)
    a3 = _rand_field((4, 9, 10), 16)
    b3 = _rand_field((5, 9, 10), 17)
    j3 = np.concatenate([a3, np.full((1, 9, 10), np.nan, np.float32), b3], axis=0)
    np.testing.assert_array_equal(oracle.ecc_hard(j3, 20, 0.0, 1.0),
                                  oracle.ecc_hard(a3, 20, 0.0, 1.0) +
                                  oracle.ecc_hard(b3, 20, 0.0, 1.0))


def test_inclusion_exclusion_over_slabs():
    """chi(A u B) = chi(A) + chi(B) - chi(A n B) for slabs sharing one plane."""
    f = _rand_field((12, 10, 11), 18)
    full = oracle.ecc_hard(f, 40, 0.0, 1.0)
    m = 5
    parts = oracle.ecc_hard(f[: m + 1], 40, 0.0, 1.0) + oracle.ecc_hard(f[m:], 40, 0.0, 1.0)
    np.testing.assert_array_equal(full, parts - oracle.ecc_hard(f[m], 40, 0.0, 1.0))
    g = _rand_field((31, 17), 19)
    full = oracle.ecc_hard(g, 40, 0.0, 1.0)
    parts = oracle.ecc_hard(g[:13], 40, 0.0, 1.0) + oracle.ecc_hard(g[12:], 40, 0.0, 1.0)
    np.testing.assert_array_equal(full, parts - oracle.ecc_hard(g[12:13], 40, 0.0, 1.0))


def test_uint8_matches_float_and_monotone_relabel():
    q = synthetic.quantise_u8(_rand_field((24, 33), 20))
    e8 = oracle.ecc_hard(q, 256, 0.0, 255.0)
    ef = oracle.ecc_hard(q.astype(np.float32), 256, 0.0, 255.0)
    np.testing.assert_array_equal(e8, ef)
    # a strictly increasing relabel applied to values and thresholds leaves the curve unchanged
    relabel = (np.arange(256, dtype=np.float64) ** 1.5 + 3.0 * np.arange(256))
    g = relabel[q].astype(np.float32)
    er = np.array([oracle.ecc_hard(g, 1, 0.0, float(np.float32(relabel[k])))[0]
                   for k in range(0, 256, 17)])
    np.testing.assert_array_equal(er, e8[::17])


def test_nan_and_out_of_range_values():
    f = _rand_field((16, 16), 21)
    g = f.copy()
    g[3, 4] = np.nan
    g[10, 10] = 7.0
    h = f.copy()
    h[3, 4] = 100.0
    h[10, 10] = 100.0
    # NaN and values above vmax never enter, exactly like a large value
    np.testing.assert_array_equal(oracle.ecc_hard(g, 32, 0.0, 1.0),
                                  oracle.ecc_hard(h, 32, 0.0, 1.0))
    lo = f.copy()
    lo[5, 5] = -np.inf
    lo2 = f.copy()
    lo2[5, 5] = -5.0
    np.testing.assert_array_equal(oracle.ecc_hard(lo, 32, 0.0, 1.0),
                                  oracle.ecc_hard(lo2, 32, 0.0, 1.0))


def test_pool_of_slabs_equals_the_whole_volume():
    """The helper that spreads the oracle over the host's cores (slabs sharing one plane, one
    process each) must give the whole volume's curve exactly, for several slab lengths."""
    from tests import _oracle_pool

    f = _rand_field((23, 9, 14), 40)
    want = oracle.ecc_hard(f, 30, 0.0, 1.0)
    for slab in (2, 3, 7, 30):
        np.testing.assert_array_equal(_oracle_pool.hard_volume(f, 30, 0.0, 1.0, slab), want)
    q = (f * 255).astype(np.uint8)
    np.testing.assert_array_equal(_oracle_pool.hard_volume(q, 256, 0.0, 255.0),
                                  oracle.ecc_hard(q, 256, 0.0, 255.0))
