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


# ---------------------------------------------------------------------------------------------
# Coded keys (the TMA-staged 3-D kernel): 1024 + 4k + (x & 1) + 2 (y & 1) as fp16 patterns,
# strict in-plane flags, and the vertical fold carried from plane to plane
# ---------------------------------------------------------------------------------------------

def coded_values(K, H, yx0=(0, 0)):
    """fp16 values of the kernel's coded key patterns 0x6400 + 4k + code (k = H, "never", gives
    0x6800 + code for H = 256: the values 2048 .. 2054)."""
    yy, xx = np.indices(K.shape[-2:])
    code = ((xx + yx0[1]) & 1) + 2 * ((yy + yx0[0]) & 1)
    pat = (0x6400 + 4 * K + code).astype(np.uint16)
    return pat.view(np.float16).astype(np.float64), pat


def c2_coded(P):
    """c2 of one plane of coded values P (padded by one with coded "never" values)."""
    Hh, Ww = P.shape[0] - 2, P.shape[1] - 2

    def nb(dy, dx):
        return P[1 + dy:1 + dy + Hh, 1 + dx:1 + dx + Ww]

    p = nb(0, 0)
    sat = lambda d: np.clip(d, 0.0, 1.0)  # the kernel's sub.sat of exact fp16 differences
    # every difference of these fp16 integers is exact, so each flag is exactly 0 or 1
    f = {k: sat(p - nb(*o)) > 0 for k, o in
         dict(W=(0, -1), E=(0, 1), S=(1, 0), NW=(-1, -1), NE=(-1, 1), SW=(1, -1),
              SE=(1, 1)).items()}
    Sp = sat(nb(-1, 0) - p) > 0
    W, E, S, NW, NE, SW, SE = (f[k] for k in ("W", "E", "S", "NW", "NE", "SW", "SE"))
    return ((Sp | (E & NE)).astype(int) - (E & ~(S & SE)) - (S & ~(W & SW)) - (W & (Sp | ~NW)))


def curve_3d_coded(K, H):
    """The TMA kernel's algebra: coded keys, strict flags, carried fold, bin = (pattern -
    0x6400) >> 2 (bin H collects the discarded "never" voxels)."""
    D, Hy, Wx = K.shape
    Kp = np.full((D + 2, Hy + 2, Wx + 2), H, np.int64)  # outside: NaN, i.e. key H
    Kp[1:-1, 1:-1, 1:-1] = K
    V, PAT = coded_values(Kp, H, yx0=(1, 1))  # padded index i is grid index i - 1
    h = np.zeros(H + 1, np.int64)
    up = lambda z: V[z + 1, 1:-1, 1:-1] < V[z, 1:-1, 1:-1]  # [k_{z+1} < k_z] (padded z)
    c2M = lambda z: c2_coded(np.maximum(V[z], V[z + 1]))
    q = -(1 - up(0)) * c2M(0)  # the plane below the volume (all never)
    for z in range(1, D + 1):
        u = up(z)
        cm = c2M(z)
        c = c2_coded(V[z]) - u * cm + q
        q = -(1 - u) * cm
        assert c.min() >= -8 and c.max() <= 7
        bins = ((PAT[z, 1:-1, 1:-1].astype(np.int64) - 0x6400) >> 2)
        np.add.at(h, np.minimum(bins, H).ravel(), c.ravel())
    return np.cumsum(h[:H])


@pytest.mark.parametrize("seed", range(3))
def test_coded_keys_and_carried_fold_match_oracle(seed):
    """Ties, NaN and every table size up to 256 (where "never" rounds above 2048)."""
    rng = np.random.default_rng(300 + seed)
    for _ in range(25):
        shp = tuple(rng.integers(1, 7, size=3))
        H = int(rng.choice([1, 2, 3, 7, 11, 255, 256]))
        img = rng.integers(0, 6, size=shp).astype(np.float32) / 5
        img[rng.random(shp) < 0.08] = np.nan
        K = keys_of(img, H, 0.0, 0.8)
        np.testing.assert_array_equal(curve_3d_coded(K, H), oracle.ecc_hard(img, H, 0.0, 0.8))
    f = synthetic.grf((12, 20, 26), 30 + seed)
    np.testing.assert_array_equal(curve_3d_coded(keys_of(f, 256, 0, 1), 256),
                                  oracle.ecc_hard(f, 256, 0, 1))


def test_coded_key_patterns():
    """Coded keys are finite fp16 integers ordered like (k, code); "never" (k = H <= 256) lies
    above every valid coded key, is an even integer when it exceeds 2048, and falls in bin H; the
    integer coding of a key pair carries nothing across halves."""
    for H in (1, 5, 200, 255, 256):
        k = np.arange(H + 1)
        for code in range(4):
            pat = 0x6400 + 4 * k + code
            val = pat.astype(np.uint16).view(np.float16).astype(np.float64)
            assert np.all(np.diff(val[:H]) > 0) and val[H] > (1024 + 4 * (H - 1) + 3)
            assert np.all(((pat - 0x6400) >> 2) == k)
            if val[H] >= 2048:
                assert val[H] % 2 == 0
    # pair coding: 4 * pair + C (mod 2^32), C = c0 + (c1 << 16) - 3 * 0x64006400
    for k0, k1, c0, c1 in [(0, 0, 0, 1), (255, 256, 2, 3), (256, 0, 0, 1), (256, 256, 2, 3)]:
        pair = (0x6400 + k0) | ((0x6400 + k1) << 16)
        C = (c0 + (c1 << 16) - 3 * 0x64006400) % 2 ** 32
        got = (4 * pair + C) % 2 ** 32
        assert got == (0x6400 + 4 * k0 + c0) | ((0x6400 + 4 * k1 + c1) << 16)


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


# ---------------------------------------------------------------------------------------------
# Soft path, 3-D: the prep kernel's local contribution from the 27 cells containing a voxel
# ---------------------------------------------------------------------------------------------

def cell_table_3d():
    """Bit masks (bit (dz+1) 9 + (dy+1) 3 + (dx+1)) of the vertices of the 27 cells containing a
    voxel, one direction in {-1, 0, +1} per axis, and their signs (-1)^dim."""
    masks, signs = [], []
    for s in range(27):
        d = (s // 9 - 1, (s // 3) % 3 - 1, s % 3 - 1)
        m = 0
        for a in range(2 if d[0] else 1):
            for b in range(2 if d[1] else 1):
                for c in range(2 if d[2] else 1):
                    m |= 1 << ((a * d[0] + 1) * 9 + (b * d[1] + 1) * 3 + (c * d[2] + 1))
        masks.append(m)
        signs.append((-1) ** sum(x != 0 for x in d))
    return masks, signs


def c3_soft_model(rank):
    """rank: the (X, linear index) order of each voxel as an integer array (absent = ABSENT)."""
    D, Hh, Ww = rank.shape
    P = np.full((D + 2, Hh + 2, Ww + 2), ABSENT, np.int64)
    P[1:-1, 1:-1, 1:-1] = rank
    earlier = np.full(rank.shape, 1 << 13, np.int64)
    for o in range(27):
        if o == 13:
            continue
        dz, dy, dx = o // 9 - 1, (o // 3) % 3 - 1, o % 3 - 1
        q = P[1 + dz:1 + dz + D, 1 + dy:1 + dy + Hh, 1 + dx:1 + dx + Ww]
        earlier |= (q < rank).astype(np.int64) << o  # ranks are distinct: < is the order
    masks, signs = cell_table_3d()
    c = np.zeros(rank.shape, np.int64)
    for m, sg in zip(masks, signs):
        c += sg * ((earlier & m) == m)
    return c


@pytest.mark.parametrize("shape,seed", [((5, 6, 7), 0), ((3, 9, 4), 1), ((1, 6, 8), 2)])
def test_soft3d_cell_table_matches_oracle(shape, seed):
    """X in fp64, order by (X, linear index), c from the 27-cell masks: sum_p c sigma(...) is the
    oracle's soft forward; quantised values make many exact ties."""
    f = np.round(synthetic.grf(shape, seed) * 7) / 7
    f = f.astype(np.float32)
    u = np.asarray([0.0, 0.05, -0.1], np.float32) if seed else np.zeros(3, np.float32)
    coords = [np.zeros(1) if n == 1 else (2.0 * np.arange(n) - (n - 1)) / (n - 1) for n in shape]
    X = f.astype(np.float64)
    for d in range(3):
        sh = [1, 1, 1]
        sh[d] = shape[d]
        X = X + np.float64(u[d]) * coords[d].reshape(sh)
    order = np.lexsort((np.arange(X.size), X.reshape(-1)))
    rank = np.empty(X.size, np.int64)
    rank[order] = np.arange(X.size)
    c = c3_soft_model(rank.reshape(shape))
    assert c.min() >= -5 and c.max() <= 7
    tau = np.linspace(-0.2, 1.2, 9).astype(np.float32)
    lam = 30.0
    s = (c.reshape(-1, 1) / (1 + np.exp(-lam * (tau.astype(np.float64) -
                                                X.reshape(-1, 1))))).sum(0)
    np.testing.assert_allclose(s, oracle.ecc_soft_fwd(f, tau, lam, 1.0, u, ndim=3), rtol=1e-11,
                               atol=1e-11)


def test_soft3d_contribution_extremes():
    """The local contribution spans [-5, 7], which the entry's 4-bit field (c + 8) holds: -5 when
    only the six axis neighbours are earlier, +7 when the 18 axis and face-diagonal neighbours
    are but no corner is."""
    r = np.full((3, 3, 3), 100, np.int64)
    r[1, 1, 1] = 50
    for z, y, x in [(0, 1, 1), (2, 1, 1), (1, 0, 1), (1, 2, 1), (1, 1, 0), (1, 1, 2)]:
        r[z, y, x] = 0
    assert c3_soft_model(r)[1, 1, 1] == -5
    dist = np.abs(np.indices((3, 3, 3)) - 1).sum(0)
    r = np.where(dist <= 2, 0, 100)
    r[1, 1, 1] = 50
    assert c3_soft_model(r)[1, 1, 1] == 7


# ---------------------------------------------------------------------------------------------
# Stencil flags from saturating fp16 subtraction (tables of at most 1024 bins)
# ---------------------------------------------------------------------------------------------

def test_saturating_flags_equal_the_comparisons_for_every_key_pair():
    """For key patterns 0x6400 + k (k <= 1024, fp16 value 1024 + k) the kernels take
    [a < p] = sat(p - a) and [a <= p] = sat((p + 1) - a). Check every pair of keys exhaustively
    in fp16 arithmetic: both are exact for every centre p with key below 1024 (a counted voxel of
    a table of at most 1024 bins), and the flags are the bit patterns 0x3C00 (1.0) / 0x0000."""
    k = np.arange(0, 1025)
    vals = (np.uint16(0x6400) + k.astype(np.uint16)).view(np.float16)
    a, p = vals[:, None], vals[None, :]
    one = np.float16(1.0)

    def sat(x):
        return np.clip(x, np.float16(0), np.float16(1)).astype(np.float16)

    lt = sat((p - a).astype(np.float16))
    le = sat(((p + one).astype(np.float16) - a).astype(np.float16))
    ka, kp = k[:, None], k[None, :]
    np.testing.assert_array_equal(lt == 1, ka < kp)
    counted = k < 1024
    np.testing.assert_array_equal((le == 1)[:, counted], (ka <= kp)[:, counted])
    assert set(np.unique(lt.view(np.uint16))) == {0, 0x3C00}
    assert set(np.unique(le.view(np.uint16))) == {0, 0x3C00}
    # beyond key 1023 the +1 is no longer exact in fp16, which is why larger tables compare
    v = (np.uint16(0x6400) + np.arange(1024, 1100).astype(np.uint16)).view(np.float16)
    assert not np.all((v + one).astype(np.float16) - v == one)


def test_fold_with_the_bias_in_the_first_product_is_exact():
    """The 3-D kernels (tables of at most 1024 bins) form 1280 + c as
    cs - fma(cn, up, fma(cm, dn, -1280)), with cs = c2(S_z), cn = c2(M_z), cm = c2(M_{z-1}) and
    the 0/1 flags up, dn. Every intermediate is an integer below 2048 in magnitude, so each fp16
    step (round to nearest) is exact; checked over every value the stencils and flags take, and
    the low byte of the result is c as a signed byte (the histogram's sign extension)."""
    f16 = np.float16
    c2_vals = np.arange(-4, 5)  # c2 of a 3 x 3 neighbourhood lies in [-3, 1]; a margin around it
    cs, cn, cm, up, dn = np.meshgrid(c2_vals, c2_vals, c2_vals, [0, 1], [0, 1], indexing="ij")
    cs, cn, cm, up, dn = (x.ravel() for x in (cs, cn, cm, up, dn))

    def h(x):
        return np.asarray(x, dtype=np.float64).astype(f16)

    t = h(h(cm) * h(dn) + h(-1280.0))     # products of small integers are exact: one rounding
    t = h(h(cn) * h(up) + t.astype(np.float64))
    res = h(h(cs).astype(np.float64) - t.astype(np.float64))
    c = cs - up * cn - dn * cm
    np.testing.assert_array_equal(res.astype(np.float64), 1280.0 + c)
    low = (res.view(np.uint16) & 0xFF).astype(np.int64)
    np.testing.assert_array_equal(np.where(low >= 128, low - 256, low), c)


def c2_neighbour_table():
    """T2[m]: the in-plane cells containing the centre of a 3 x 3 patch, summed with signs
    (-1)^dim over the cells whose other vertices are all in the 8-bit neighbour mask m (bits
    0..7: (dy, dx) = (-1,-1), (-1,0), (-1,1), (0,-1), (0,1), (1,-1), (1,0), (1,1))."""
    nb = [(dy, dx) for dy in (-1, 0, 1) for dx in (-1, 0, 1) if (dy, dx) != (0, 0)]
    bit = {d: i for i, d in enumerate(nb)}
    t = np.zeros(256, np.int64)
    for m in range(256):
        v = 0
        for sy in (-1, 0, 1):
            for sx in (-1, 0, 1):
                need = 0
                for a in range(2 if sy else 1):
                    for b in range(2 if sx else 1):
                        if (a * sy, b * sx) != (0, 0):
                            need |= 1 << bit[(a * sy, b * sx)]
                if m & need == need:
                    v += (-1) ** ((sy != 0) + (sx != 0))
        t[m] = v
    return t


def test_slice_fold_of_the_27_cells_in_bits():
    """The 3-D soft prep forms c3 from the 26-bit 'earlier' mask as
        c3 = T2[m0] - e_below T2[m0 & m_below] - e_above T2[m0 & m_above],
    with m0, m_below, m_above the 8 neighbour bits of the planes z, z - 1, z + 1 and e_below,
    e_above the voxels straight below and above (the slice fold of the hard path, in bits). The
    27 cells split into those of plane z, those reaching z - 1 and those reaching z + 1, so it
    suffices to check every (plane z, plane z - 1) mask pair with plane z + 1 empty and every
    (plane z, plane z + 1) pair with plane z - 1 empty: 2 x 2^17 masks, all of them."""
    masks, signs = cell_table_3d()
    t2 = c2_neighbour_table()

    def compress9(x):  # 9 plane bits without the centre (bit 4) -> 8 bits
        return (x & 0xF) | ((x >> 1) & 0xF0)

    def expand8(m):  # 8 neighbour bits -> 9 plane bits with the centre bit clear
        return (m & 0xF) | ((m & 0xF0) << 1)

    m0 = np.repeat(np.arange(256, dtype=np.int64), 512)
    other = np.tile(np.arange(512, dtype=np.int64), 256)
    for shift in (0, 18):  # plane z - 1 or plane z + 1 populated
        earlier = (expand8(m0) << 9) | (1 << 13) | (other << shift)
        want = np.zeros(earlier.shape, np.int64)
        for m, sg in zip(masks, signs):
            want += sg * ((earlier & m) == m)
        xb, xa = earlier & 0x1FF, (earlier >> 18) & 0x1FF
        mz = compress9((earlier >> 9) & 0x1FF)
        got = (t2[mz] - ((xb >> 4) & 1) * t2[mz & compress9(xb)]
               - ((xa >> 4) & 1) * t2[mz & compress9(xa)])
        np.testing.assert_array_equal(got, want)
    # the table is the 2-D local contribution: its range is [-3, 1]
    assert t2.min() == -3 and t2.max() == 1
