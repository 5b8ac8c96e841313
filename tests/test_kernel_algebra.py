"""The algebra the hard-ECC kernels implement, checked in numpy against the oracle (CPU only).

The kernels compute, per pixel, the local Euler contribution on (key, linear index) order with
the identity
    c = (Sp | E NE) - E ~(S SE) - S ~(W SW) - W (Sp | ~NW),     Sp = "pixel above not earlier",
and in 3-D fold the max-slice terms into the voxel that carries them:
    c3(p) = c2(S_z; p) - [k_{z+1} < k_z] c2(M_z) - [k_{z-1} <= k_z] c2(M_{z-1}).
Contributions travel as the fp16 value 1280 + c, whose low pattern byte is c. These tests
restate that algebra with numpy integers and check the resulting curves against the oracle.
"""
import numpy as np
import pytest

import oracle
from euler_characteristic_curves_gb300 import synthetic

ABSENT = 10 ** 9


def keys_of(img, H, vmin, vmax):
    t = oracle.thresholds(H, vmin, vmax)
    k = np.searchsorted(t, img.astype(np.float64), side="left")  # first k with v <= t_k
    k[np.isnan(img)] = H
    return k.astype(np.int64)


def c2_kernel(K):
    Hh, Ww = K.shape
    P = np.full((Hh + 2, Ww + 2), ABSENT, np.int64)
    P[1:-1, 1:-1] = K

    def nb(dy, dx):
        return P[1 + dy:1 + dy + Hh, 1 + dx:1 + dx + Ww]

    p = K
    W, E, S = nb(0, -1) <= p, nb(0, 1) < p, nb(1, 0) < p
    NW, NE = nb(-1, -1) <= p, nb(-1, 1) <= p
    SW, SE = nb(1, -1) < p, nb(1, 1) < p
    Sp = p < nb(-1, 0)
    return ((Sp | (E & NE)).astype(int) - (E & ~(S & SE)) - (S & ~(W & SW)) - (W & (Sp | ~NW)))


def curve_2d(K, H):
    c = c2_kernel(K)
    h = np.zeros(H + 1, np.int64)
    m = (c != 0) & (K < H)
    np.add.at(h, K[m], c[m])
    return np.cumsum(h[:H])


def curve_3d(K, H):
    D = K.shape[0]
    h = np.zeros(H + 1, np.int64)
    pad = np.full((D + 2,) + K.shape[1:], ABSENT, np.int64)
    pad[1:-1] = K
    for z in range(D):
        cur, nxt, prv = pad[z + 1], pad[z + 2], pad[z]
        c = (c2_kernel(cur) - (nxt < cur) * c2_kernel(np.maximum(cur, nxt))
             - (prv <= cur) * c2_kernel(np.maximum(prv, cur)))
        assert c.min() >= -8 and c.max() <= 7  # fits the 1280 + c byte encoding
        m = (c != 0) & (cur < H)
        np.add.at(h, cur[m], c[m])
    return np.cumsum(h[:H])


@pytest.mark.parametrize("seed", range(4))
def test_2d_identity_matches_oracle(seed):
    rng = np.random.default_rng(seed)
    for _ in range(40):
        shp = tuple(rng.integers(1, 10, size=2))
        H = int(rng.integers(1, 12))
        img = rng.integers(0, 6, size=shp).astype(np.float32) / 5
        img[rng.random(shp) < 0.08] = np.nan
        K = keys_of(img, H, 0.0, 0.8)
        np.testing.assert_array_equal(curve_2d(K, H), oracle.ecc_hard(img, H, 0.0, 0.8))


@pytest.mark.parametrize("seed", range(3))
def test_3d_fold_matches_oracle(seed):
    rng = np.random.default_rng(100 + seed)
    for _ in range(25):
        shp = tuple(rng.integers(1, 7, size=3))
        H = int(rng.integers(1, 12))
        img = rng.integers(0, 6, size=shp).astype(np.float32) / 5
        img[rng.random(shp) < 0.08] = np.nan
        K = keys_of(img, H, 0.0, 0.8)
        np.testing.assert_array_equal(curve_3d(K, H), oracle.ecc_hard(img, H, 0.0, 0.8))
    f = synthetic.grf((20, 24, 28), 3 + seed)
    np.testing.assert_array_equal(curve_3d(keys_of(f, 256, 0, 1), 256),
                                  oracle.ecc_hard(f, 256, 0, 1))


def test_key_patterns_and_contribution_encoding():
    # 0x6400 + k is a strictly increasing fp16 pattern for k <= 6143, below +inf (absent)
    k = np.arange(0, 6144)
    vals = (0x6400 + k).astype(np.uint16).view(np.float16).astype(np.float64)
    assert np.all(np.diff(vals) > 0) and np.all(np.isfinite(vals))
    assert np.float16(np.inf).view(np.uint16) == 0x7C00 > 0x6400 + 6143
    # 1280 + c has pattern 0x6500 + c, whose low byte is c as a signed byte
    for c in range(-8, 8):
        pat = int(np.float16(1280 + c).view(np.uint16))
        assert pat == 0x6500 + c and np.array(pat & 0xFF, np.uint8).view(np.int8) == c
