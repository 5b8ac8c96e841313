"""The hard and soft ECC sharded over ranks (one GPU per rank), with one all-reduce per call.

Paper notes "Scalable GPU-Accelerated Euler Characteristic Curves: Optimization and
Differentiable Learning for PyTorch", section "Limitations": the method runs on one device,
without batching or multi-GPU execution. The ECC is a sum over the cells of the grid, each cell
counted at the bin where its largest vertex enters, so per-bin counts add over pieces that share
no cells:

* a batch splits by images (no cell joins two images), and the soft gradients with respect to
  the shared tau, alpha and u are sums over the images;
* one volume splits into slabs of planes in which consecutive slabs share one plane. Every cell
  spans at most two consecutive planes, so it lies in some slab, and two consecutive slabs share
  exactly the cells of their common plane:
      hist(volume) = sum_r hist_3D(slab r) - sum_{r > 0} hist_2D(first plane of slab r).

Each rank computes its partial histogram with ``ecc_hard_partial`` (no running sum), the ranks
sum them with one all-reduce of nbins int64 per image, and the running sum ``hist_to_curve`` gives
the curve that ``ecc_hard`` returns for the whole grid. The soft path sums its per-rank gradients
(K + 1 + ndim floats) and the zero-padded rows of S in one all-reduce of a float buffer.

The plans (``slab_plan``, ``batch_plan``) are host logic. The per-rank compute, the all-reduce and
the running sum are arguments with library defaults (``torch.distributed.all_reduce`` on the
default group), so the same exchange runs under NCCL on GPUs, under gloo on CPU, or as virtual
ranks in one process that sum into one buffer.
"""
from __future__ import annotations

import torch


def slab_plan(depth: int, world: int) -> list[tuple[int, int]]:
    """Planes [a_r, b_r] (inclusive) of rank r's slab for a volume of ``depth`` planes: a_0 = 0,
    b_{world-1} = depth - 1 and a_{r+1} = b_r (consecutive slabs share one plane); the cuts are
    spread evenly. With fewer planes than ranks some slabs are a single shared plane, which adds
    and subtracts the same cells (their rank contributes nothing)."""
    if depth < 1 or world < 1:
        raise ValueError("depth and world must be positive")
    cuts = [round(r * (depth - 1) / world) for r in range(world + 1)]
    return [(cuts[r], cuts[r + 1]) for r in range(world)]


def batch_plan(batch: int, world: int) -> list[tuple[int, int]]:
    """Images [lo_r, hi_r) of rank r: contiguous, sizes differing by at most one."""
    if batch < 1 or world < 1:
        raise ValueError("batch and world must be positive")
    return [(r * batch // world, (r + 1) * batch // world) for r in range(world)]


def _library_partial(x, nbins, vmin, vmax, sign, hist, ndim):
    from . import ecc

    ecc.ecc_hard_partial(x, nbins, vmin, vmax, hist, sign=sign, ndim=ndim)


def _library_curve(hist):
    from . import ecc

    ecc.hist_to_curve(hist)


def _default_allreduce(group):
    import torch.distributed as dist

    def reduce(t):
        if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
            dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
        return t

    return reduce


def volume_partial(slab: torch.Tensor, nbins: int, vmin: float, vmax: float, rank: int,
                   hist: torch.Tensor, partial=None) -> torch.Tensor:
    """Adds rank ``rank``'s share of a volume's histogram into ``hist`` (int64 [nbins]): + the
    cells of its slab ([planes, H, W], the planes of ``slab_plan``), - the cells of the slab's
    first plane when a previous rank holds it too (rank > 0)."""
    partial = partial or _library_partial
    partial(slab, nbins, vmin, vmax, +1, hist, 3)
    if rank > 0:
        partial(slab[0], nbins, vmin, vmax, -1, hist, 2)
    return hist


def ecc_hard_volume_sharded(slab: torch.Tensor, nbins: int, vmin: float, vmax: float, rank: int,
                            group=None, partial=None, allreduce=None,
                            to_curve=None) -> torch.Tensor:
    """Hard ECC (int64 [nbins], on every rank) of a volume whose slabs of ``slab_plan`` are spread
    over the ranks; ``slab`` is this rank's. One all-reduce of nbins int64."""
    hist = torch.zeros(nbins, dtype=torch.int64, device=slab.device)
    volume_partial(slab, nbins, vmin, vmax, rank, hist, partial)
    (allreduce or _default_allreduce(group))(hist)
    (to_curve or _library_curve)(hist)
    return hist


def ecc_hard_batch_sharded(images: torch.Tensor, lo: int, batch: int, nbins: int, vmin: float,
                           vmax: float, ndim: int, group=None, partial=None, allreduce=None,
                           to_curve=None) -> torch.Tensor:
    """Hard ECC (int64 [batch, nbins], on every rank) of a batch whose images [lo, lo + n) are
    this rank's (``images``: [n, (D,) H, W], the ranges of ``batch_plan``). One all-reduce of
    batch * nbins int64."""
    hist = torch.zeros((batch, nbins), dtype=torch.int64, device=images.device)
    n = images.shape[0]
    if n > 0:
        (partial or _library_partial)(images, nbins, vmin, vmax, +1, hist[lo:lo + n], ndim)
    (allreduce or _default_allreduce(group))(hist)
    (to_curve or _library_curve)(hist)
    return hist


def _library_soft(images, tau, lam, alpha, u, grad_out, ndim):
    from . import ecc

    s, ws = ecc.ecc_soft_fwd(images, tau, lam, alpha, u, ndim=ndim)
    if grad_out is None:
        return s, None
    g = ecc.ecc_soft_bwd(images, tau, lam, alpha, u, grad_out, ws, ndim=ndim)
    return s, (g["grad_tau"], g["grad_alpha"], g["grad_u"])


def soft_ecc_batch_sharded(images: torch.Tensor, lo: int, batch: int, tau: torch.Tensor,
                           lam: float, alpha: torch.Tensor, u: torch.Tensor,
                           grad_out: torch.Tensor | None = None, ndim: int | None = None,
                           group=None, local=None, allreduce=None):
    """Soft ECC of a batch whose images [lo, lo + n) are this rank's, with the gradients of
    sum(grad_out * S) when this rank's upstream gradient rows ``grad_out`` ([n, K]) are given.

    Returns (S [batch, K], grads or None) on every rank, grads = (grad_tau [K], grad_alpha [1],
    grad_u [ndim]) summed over all images. One all-reduce of batch * K + K + 1 + ndim floats:
    S rows of other ranks are zero here and exact after the sum."""
    ndim = u.numel() if ndim is None else ndim
    K = tau.numel()
    n = images.shape[0]
    buf = torch.zeros(batch * K + K + 1 + ndim, dtype=torch.float32, device=images.device)
    if n > 0:
        s, grads = (local or _library_soft)(images, tau, lam, alpha, u, grad_out, ndim)
        buf[lo * K:(lo + n) * K] = s.reshape(-1)
        if grads is not None:
            gt, ga, gu = grads
            tail = buf[batch * K:]
            tail[:K] = gt.reshape(-1)
            tail[K] = ga.reshape(-1)[0]
            tail[K + 1:] = gu.reshape(-1)
    (allreduce or _default_allreduce(group))(buf)
    S = buf[:batch * K].view(batch, K)
    if grad_out is None:
        return S, None
    tail = buf[batch * K:]
    return S, (tail[:K], tail[K:K + 1], tail[K + 1:])
