"""Seeded synthetic inputs shaped like the workloads of the ECC paper notes' timing tables
("Key experimental data": 2-D grids 128^2 .. 8192^2, 3-D grids 128^3 .. 1024^3, synthetic grids).

This module only draws random numbers and shapes them; it holds none of the Euler-characteristic
arithmetic, so the CUDA path, the CPU oracle and the benchmark can all take their inputs from it.

Recipes:
  * grf: Gaussian random field with power spectrum ~ |k|^-slope (slope 3 by default).
    White N(0, 1) noise -> real FFT -> multiply by |k|^(-slope/2) with integer frequencies and the
    DC term set to 0 -> inverse FFT (periodic field) -> min-max normalised to [0, 1] -> float32.
  * blurred_noise_u8: white N(0, 1) noise -> periodic Gaussian blur (sigma in pixels, applied in
    Fourier space) -> min-max normalised -> round(255 v) as uint8.
  * quantise_u8: round(255 v) of a [0, 1] field, as uint8.
  * soft_direction / upstream_grad: u ~ N(0, sigma_u^2) per axis; dL/dECC ~ N(0, 1).

CPU generation uses numpy's PCG64 (np.random.default_rng(seed)); CUDA generation uses torch's
Philox generator seeded with the same seed (different streams of numbers: a test or a benchmark
generates once and gives the same bytes to every consumer).
"""
from __future__ import annotations

import numpy as np


def _freq_sq_numpy(shape, real_last: bool):
    axes = []
    for i, n in enumerate(shape):
        if real_last and i == len(shape) - 1:
            axes.append(np.fft.rfftfreq(n) * n)
        else:
            axes.append(np.fft.fftfreq(n) * n)
    grids = np.meshgrid(*axes, indexing="ij", sparse=True)
    k2 = np.zeros([len(a) for a in axes], np.float64)
    for g in grids:
        k2 = k2 + g * g
    return k2


def grf(shape, seed: int, slope: float = 3.0, batch: int | None = None, device: str = "cpu"):
    """Float32 Gaussian random field(s) in [0, 1] of the given spatial shape.

    Returns a numpy array on device "cpu", a torch tensor on a CUDA device. With ``batch`` the
    result has a leading batch axis; each image is generated and normalised independently.
    """
    shape = tuple(int(s) for s in shape)
    if device != "cpu":
        return _grf_torch(shape, seed, slope, batch, device)
    rng = np.random.default_rng(seed)
    nb = 1 if batch is None else int(batch)
    k2 = _freq_sq_numpy(shape, real_last=True)
    k2.flat[0] = 1.0
    amp = k2 ** (-slope / 4.0)
    amp.flat[0] = 0.0
    out = np.empty((nb,) + shape, np.float32)
    for b in range(nb):
        w = rng.standard_normal(shape)
        ax = list(range(len(shape)))
        f = np.fft.irfftn(np.fft.rfftn(w, axes=ax) * amp, s=shape, axes=ax)
        lo, hi = f.min(), f.max()
        out[b] = ((f - lo) / (hi - lo)).astype(np.float32)
    return out if batch is not None else out[0]


def _grf_torch(shape, seed, slope, batch, device):
    import torch

    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    nb = 1 if batch is None else int(batch)
    axes = []
    for i, n in enumerate(shape):
        if i == len(shape) - 1:
            f = torch.fft.rfftfreq(n, device=device) * n
        else:
            f = torch.fft.fftfreq(n, device=device) * n
        axes.append(f.to(torch.float32))
    out = torch.empty((nb,) + shape, dtype=torch.float32, device=device)
    for b in range(nb):
        w = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        F = torch.fft.rfftn(w)
        del w
        k2 = None
        for i, a in enumerate(axes):
            view = [1] * len(shape)
            view[i] = a.numel()
            term = (a * a).view(view)
            k2 = term if k2 is None else k2 + term
        k2 = k2.clone()
        k2.view(-1)[0] = 1.0
        amp = k2.pow_(-slope / 4.0)
        amp.view(-1)[0] = 0.0
        F.mul_(amp)
        del amp, k2
        f = torch.fft.irfftn(F, s=shape)
        del F
        lo, hi = f.min(), f.max()
        out[b] = (f - lo) / (hi - lo)
        del f
    return out if batch is not None else out[0]


def blurred_noise_u8(shape, seed: int, sigma: float = 3.0):
    """uint8 image: periodic Gaussian blur (sigma px) of white noise, min-max, round(255 v)."""
    shape = tuple(int(s) for s in shape)
    rng = np.random.default_rng(seed)
    w = rng.standard_normal(shape)
    axes = [np.fft.fftfreq(n) for n in shape[:-1]] + [np.fft.rfftfreq(shape[-1])]
    grids = np.meshgrid(*axes, indexing="ij", sparse=True)
    k2 = sum(g * g for g in grids)
    # Fourier transform of a unit-mass Gaussian of std sigma (frequencies in cycles per pixel)
    kernel = np.exp(-2.0 * (np.pi * sigma) ** 2 * k2)
    ax = list(range(len(shape)))
    f = np.fft.irfftn(np.fft.rfftn(w, axes=ax) * kernel, s=shape, axes=ax)
    v = (f - f.min()) / (f.max() - f.min())
    return np.rint(255.0 * v).astype(np.uint8)


def quantise_u8(v):
    """round(255 v) as uint8 for a [0, 1] float field (numpy array or torch tensor)."""
    if isinstance(v, np.ndarray):
        return np.rint(255.0 * v.astype(np.float64)).astype(np.uint8)
    import torch

    return torch.round(v * 255.0).to(torch.uint8)


def soft_direction(ndim: int, seed: int, sigma_u: float = 0.1):
    """Direction u ~ N(0, sigma_u^2) per axis, float32."""
    rng = np.random.default_rng(seed)
    return (sigma_u * rng.standard_normal(ndim)).astype(np.float32)


def upstream_grad(shape, seed: int):
    """dL/dECC ~ N(0, 1), float32."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal(tuple(shape)).astype(np.float32)


def uniform_thresholds(K: int, lo: float = 0.0, hi: float = 1.0):
    """K soft thresholds tau_k = lo + (hi - lo) k / (K - 1), float32."""
    if K == 1:
        return np.asarray([hi], np.float32)
    return (lo + (hi - lo) * np.arange(K, dtype=np.float64) / (K - 1)).astype(np.float32)
