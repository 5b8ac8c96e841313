"""Independent topology used to pin the oracle: Betti numbers of binary grids.

Nothing here counts cells with signs; it computes connectivity (flood fill through
scipy.ndimage.label) and GF(2) homology ranks, both textbook routines, so that a wrong cell set
or sign in the oracle's Euler-characteristic sum shows up as a mismatch with
chi = b0 - b1 + b2.

For the V-construction (every voxel a vertex, boxes of side 0 or 1 as cells, a cell present when
all its corners are present) the foreground is 4-connected in 2-D and 6-connected in 3-D, and the
complement is 8- resp. 26-connected.
"""
from __future__ import annotations

import itertools

import numpy as np
from scipy import ndimage


def _conn(ndim: int, full: bool):
    return ndimage.generate_binary_structure(ndim, ndim if full else 1)


def b0(mask: np.ndarray) -> int:
    """Connected components of the foreground (axis adjacency)."""
    _, n = ndimage.label(mask, structure=_conn(mask.ndim, full=False))
    return int(n)


def cavities(mask: np.ndarray) -> int:
    """Components of the complement (full adjacency) that do not reach the grid border.

    In 2-D these are the holes (b1); in 3-D the enclosed cavities (b2).
    """
    padded = np.pad(~mask.astype(bool), 1, constant_values=True)
    lab, n = ndimage.label(padded, structure=_conn(mask.ndim, full=True))
    outside = lab[(0,) * mask.ndim]
    return int(n - (1 if outside > 0 else 0))


def chi_2d_flood(mask: np.ndarray) -> int:
    return b0(mask) - cavities(mask)


# ---------------------------------------------------------------------------------------------
# GF(2) homology of the V-construction complex of a binary 3-D grid
# ---------------------------------------------------------------------------------------------

def _cells(mask: np.ndarray):
    """Cells as frozensets of voxel coordinates, grouped by dimension."""
    nd = mask.ndim
    shape = mask.shape
    by_dim = [[] for _ in range(nd + 1)]
    for p in itertools.product(*[range(n) for n in shape]):
        for axes in itertools.product((0, 1), repeat=nd):
            if any(p[d] + axes[d] >= shape[d] for d in range(nd)):
                continue
            verts = []
            for off in itertools.product(*[((0, 1) if axes[d] else (0,)) for d in range(nd)]):
                verts.append(tuple(p[d] + off[d] for d in range(nd)))
            if all(mask[v] for v in verts):
                by_dim[sum(axes)].append((p, axes))
    return by_dim


def _faces(cell):
    """The codimension-1 faces of a box cell (lower corner, axis flags)."""
    p, axes = cell
    out = []
    for d, a in enumerate(axes):
        if not a:
            continue
        lower = list(axes)
        lower[d] = 0
        out.append((p, tuple(lower)))
        q = list(p)
        q[d] += 1
        out.append((tuple(q), tuple(lower)))
    return out


def _rank_gf2(rows):
    """Rank over GF(2) of a list of Python-int bit rows."""
    basis = {}
    rank = 0
    for r in rows:
        while r:
            top = r.bit_length() - 1
            if top in basis:
                r ^= basis[top]
            else:
                basis[top] = r
                rank += 1
                break
    return rank


def betti(mask: np.ndarray):
    """Betti numbers (b0, ..., b_ndim) over GF(2) of the V-construction complex of mask."""
    by_dim = _cells(mask)
    index = [{c: i for i, c in enumerate(cs)} for cs in by_dim]
    ranks = [0] * (len(by_dim) + 1)  # ranks[k] = rank of boundary C_k -> C_{k-1}
    for k in range(1, len(by_dim)):
        rows = []
        for c in by_dim[k]:
            r = 0
            for f in _faces(c):
                r |= 1 << index[k - 1][f]
            rows.append(r)
        ranks[k] = _rank_gf2(rows)
    return [len(by_dim[k]) - ranks[k] - ranks[k + 1] for k in range(len(by_dim))]
