"""The oracle on every host core, for full-size parity checks (test infrastructure).

The oracle is plain single-threaded C. For the full-size workloads the tests cut the work into
independent pieces and run one oracle process per host core; the pieces are combined with
identities the oracle tests pin on their own:

* a 3-D volume as slabs of planes in which consecutive slabs share one plane: every cell lies in
  some slab and two consecutive slabs share exactly the cells of their common plane, so
  ECC(volume) = sum_i ECC(slab i) - sum_{i>0} ECC(first plane of slab i) at every threshold
  (pinned on the oracle by test_inclusion_exclusion_over_slabs);
* a batch of images image by image: no cell joins two images, and the gradients with respect to
  the shared tau, alpha and u sum over the images (pinned by test_batch_is_a_sum).

Pools start with 'spawn', so no worker inherits the parent's CUDA context. A volume reaches the
workers through a temporary file that each worker maps read-only.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import tempfile
from concurrent.futures import ProcessPoolExecutor

import numpy as np


def cores() -> int:
    return max(1, min(os.cpu_count() or 1, 64))


def _pool(n_tasks: int) -> ProcessPoolExecutor:
    import oracle

    oracle.build()  # compile once, before the workers load it
    return ProcessPoolExecutor(max(1, min(cores(), n_tasks)), mp_context=mp.get_context("spawn"))


def _hard_piece(task):
    path, shape, dtype, a, b, nbins, vmin, vmax, sign = task
    import oracle

    vol = np.memmap(path, dtype=dtype, mode="r", shape=shape)
    piece = np.ascontiguousarray(vol[a] if a == b else vol[a: b + 1])
    return sign * oracle.ecc_hard(piece, nbins, vmin, vmax).astype(np.int64)


def hard_volume(vol: np.ndarray, nbins: int, vmin: float, vmax: float,
                slab_planes: int | None = None) -> np.ndarray:
    """Oracle ECC (int64 [nbins]) of one [D, H, W] volume, computed as slabs that share one plane,
    one oracle process per host core."""
    vol = np.ascontiguousarray(vol)
    D = vol.shape[0]
    if slab_planes is None:  # about three slabs per core, at least two planes each
        slab_planes = max(2, -(-D // (3 * cores())) + 1)
    cuts = [0]
    while cuts[-1] < D - 1:
        cuts.append(min(cuts[-1] + slab_planes - 1, D - 1))
    fd, path = tempfile.mkstemp(suffix=".raw")
    os.close(fd)
    try:
        vol.tofile(path)
        common = (path, vol.shape, vol.dtype.str)
        tasks = [common + (a, b, nbins, vmin, vmax, 1) for a, b in zip(cuts[:-1], cuts[1:])]
        tasks += [common + (c, c, nbins, vmin, vmax, -1) for c in cuts[1:-1]]
        if len(cuts) == 1:  # a single plane
            tasks = [common + (0, 0, nbins, vmin, vmax, 1)]
        # the largest pieces first, so the pool's tail is short
        tasks.sort(key=lambda t: t[3] - t[4])
        with _pool(len(tasks)) as ex:
            parts = list(ex.map(_hard_piece, tasks))
    finally:
        os.unlink(path)
    return np.sum(parts, axis=0)


def _soft_image(task):
    img, tau, lam, alpha, u, g, ndim, want_img = task
    import oracle

    s = oracle.ecc_soft_fwd(img, tau, lam, alpha, u, ndim=ndim)
    r = oracle.ecc_soft_bwd(img, tau, lam, alpha, u, g, ndim=ndim, want_img=want_img)
    return s, r


def soft_batch(img: np.ndarray, tau, lam, alpha, u, g, ndim: int, want_img: bool = True):
    """Oracle soft ECC and gradients of a batch [B, ...], one image per task on every core.
    Returns (S [B, K], dict as oracle.ecc_soft_bwd returns for the whole batch)."""
    B = img.shape[0]
    g = np.asarray(g, np.float64).reshape(B, -1)
    tasks = [(np.ascontiguousarray(img[b]), tau, lam, alpha, u, g[b], ndim, want_img)
             for b in range(B)]
    with _pool(B) as ex:
        res = list(ex.map(_soft_image, tasks))
    S = np.stack([s for s, _ in res])
    out = {"grad_tau": np.sum([r["grad_tau"] for _, r in res], axis=0),
           "grad_alpha": float(np.sum([r["grad_alpha"] for _, r in res])),
           "grad_u": np.sum([r["grad_u"] for _, r in res], axis=0)}
    if want_img:
        out["grad_img"] = np.stack([r["grad_img"] for _, r in res])
        out["grad_img_absterms"] = np.stack([r["grad_img_absterms"] for _, r in res])
    return S, out
