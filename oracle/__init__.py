"""CPU oracle for the Euler characteristic curve and its soft (sigmoid-relaxed) form.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``. The product path (the CUDA library
and its binding in ``euler_characteristic_curves_gb300``) never imports this package.

The arithmetic lives in ``ecc_oracle.c`` (plain C, fp64, compiled with ``-ffp-contract=off``);
this module compiles it with gcc on first use and marshals numpy arrays through ctypes. Every
function cites the passage it follows in the C source's header: the paper notes "Scalable
GPU-Accelerated Euler Characteristic Curves: Optimization and Differentiable Learning for
PyTorch", sections "Key designs -- differentiable ECC layer (sigmoid relaxation)" and
"Key designs -- local computation of the Euler characteristic coefficient".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ecc_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libecc_oracle.so")
_lock = threading.Lock()
_lib = None

U8, F32 = 0, 1


def build(force: bool = False) -> str:
    """Compile ecc_oracle.c into oracle/_build/libecc_oracle.so (plain gcc, no CUDA)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p, i64, d, i = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double, ctypes.c_int
            lib.oracle_thresholds.argtypes = [i, d, d, p]
            lib.oracle_ecc_hard.argtypes = [p, i, i, p, i64, i, d, d, p]
            lib.oracle_ecc_soft_fwd.argtypes = [p, i, p, i64, p, i, d, d, p, p]
            lib.oracle_ecc_soft_bwd.argtypes = [p, i, p, i64, p, i, d, d, p, p, p, p, p, p, p, p]
            for fn in (lib.oracle_thresholds, lib.oracle_ecc_hard, lib.oracle_ecc_soft_fwd,
                       lib.oracle_ecc_soft_bwd):
                fn.restype = i
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with status {rc}")


def thresholds(nbins: int, vmin: float, vmax: float) -> np.ndarray:
    """The nbins fp64 thresholds t_k of the hard ECC."""
    tau = np.empty(nbins, np.float64)
    _check(_load().oracle_thresholds(int(nbins), float(vmin), float(vmax), _ptr(tau)),
           "thresholds")
    return tau


def _split_batch(img: np.ndarray, ndim: int):
    if img.ndim == ndim:
        return 1, img.shape
    if img.ndim == ndim + 1:
        return img.shape[0], img.shape[1:]
    raise ValueError(f"expected a {ndim}-D image or a batch of them, got shape {img.shape}")


def ecc_hard(img: np.ndarray, nbins: int, vmin: float, vmax: float, ndim: int | None = None):
    """Hard ECC, int64 [batch, nbins] (or [nbins] for an unbatched image).

    img: uint8 or float32 array, [(B,) (D,) H, W]; ``ndim`` (2 or 3) says how many trailing axes
    form one image (default: all axes when img.ndim <= 3 -- pass it for batches of 2-D images).
    """
    img = np.ascontiguousarray(img)
    if img.dtype == np.uint8:
        dt = U8
    elif img.dtype == np.float32:
        dt = F32
    else:
        raise TypeError(f"oracle.ecc_hard: dtype {img.dtype} (uint8 or float32 expected)")
    if ndim is None:
        ndim = img.ndim
    batch, dims = _split_batch(img, ndim)
    dims_a = np.asarray(dims, np.int64)
    out = np.empty((batch, nbins), np.int64)
    _check(_load().oracle_ecc_hard(_ptr(img), dt, ndim, _ptr(dims_a), batch, int(nbins),
                                   float(vmin), float(vmax), _ptr(out)), "ecc_hard")
    return out if img.ndim == ndim + 1 else out[0]


def _soft_args(img, tau, u, ndim):
    img = np.ascontiguousarray(img, dtype=np.float32)
    tau = np.ascontiguousarray(tau, dtype=np.float32)
    if ndim is None:
        ndim = img.ndim
    batch, dims = _split_batch(img, ndim)
    u = np.ascontiguousarray(np.asarray(u, np.float32).astype(np.float64))
    if u.shape != (ndim,):
        raise ValueError(f"u must have {ndim} entries")
    return img, tau, u, ndim, batch, np.asarray(dims, np.int64)


def ecc_soft_fwd(img, tau, lam, alpha, u, ndim=None):
    """Soft ECC S[b, k] in fp64. img float32 [(B,) (D,) H, W]; tau [K]; alpha scalar; u [ndim].

    lam, alpha and u are taken as float32 values promoted to fp64 (the library's argument types).
    """
    img, tau, u, ndim, batch, dims = _soft_args(img, tau, u, ndim)
    K = tau.shape[0]
    out = np.empty((batch, K), np.float64)
    lam64 = float(np.float32(lam))
    alpha64 = float(np.float32(alpha))
    _check(_load().oracle_ecc_soft_fwd(_ptr(img), ndim, _ptr(dims), batch, _ptr(tau), K, lam64,
                                       alpha64, _ptr(u), _ptr(out)), "ecc_soft_fwd")
    return out if img.ndim == ndim + 1 else out[0]


def ecc_soft_bwd(img, tau, lam, alpha, u, grad_out, ndim=None, want_img=True):
    """Analytic gradients of sum(grad_out * S). Returns a dict of fp64 arrays:
    grad_tau [K], grad_tau_absterms [K] (the sum of |terms| that make up each grad_tau entry),
    grad_alpha (scalar), grad_u [ndim], and when want_img: grad_img (img's shape) and
    grad_img_absterms (same shape; the sum of |terms| that make up each grad_img entry)."""
    img, tau, u, ndim, batch, dims = _soft_args(img, tau, u, ndim)
    K = tau.shape[0]
    go = np.ascontiguousarray(np.asarray(grad_out, np.float64).reshape(batch, K))
    gt = np.empty(K, np.float64)
    ga = np.empty(1, np.float64)
    gu = np.empty(ndim, np.float64)
    gi = np.empty(img.shape, np.float64) if want_img else None
    gabs = np.empty(img.shape, np.float64) if want_img else None
    gtabs = np.empty(K, np.float64)
    lam64 = float(np.float32(lam))
    alpha64 = float(np.float32(alpha))
    _check(_load().oracle_ecc_soft_bwd(_ptr(img), ndim, _ptr(dims), batch, _ptr(tau), K, lam64,
                                       alpha64, _ptr(u), _ptr(go), _ptr(gt), _ptr(ga), _ptr(gu),
                                       _ptr(gi), _ptr(gabs), _ptr(gtabs)), "ecc_soft_bwd")
    res = {"grad_tau": gt, "grad_alpha": float(ga[0]), "grad_u": gu, "grad_tau_absterms": gtabs}
    if want_img:
        res["grad_img"] = gi
        res["grad_img_absterms"] = gabs
    return res


# ---------------------------------------------------------------------------------------------
# Soft Euler characteristic transform: the soft ECC along each of several directions
# ---------------------------------------------------------------------------------------------
# Paper notes "Scalable GPU-Accelerated Euler Characteristic Curves", "Limitations": the layer
# works on one direction at a time, while the Euler characteristic transform integrates the
# curve over many directions. By definition the transform's value for direction u_j is the
# (soft) ECC of the filtration X_j = alpha f + u_j . x, so the oracle evaluates the pinned
# single-direction soft ECC once per direction.

def _directions(U, ndim):
    U = np.asarray(U, np.float32)
    if U.ndim != 2 or U.shape[1] != ndim:
        raise ValueError(f"directions must have shape [n_dirs, {ndim}]")
    return U


def ecc_soft_ect_fwd(img, tau, lam, alpha, U, ndim=None):
    """S[b, j, k] = soft ECC of image b along direction U[j] (fp64); [(B,) n_dirs, K]."""
    nd = np.asarray(img).ndim if ndim is None else ndim
    U = _directions(U, nd)
    per = [ecc_soft_fwd(img, tau, lam, alpha, U[j], ndim=nd) for j in range(U.shape[0])]
    return np.stack(per, axis=-2)


def ecc_soft_ect_bwd(img, tau, lam, alpha, U, grad_out, ndim=None, want_img=True):
    """Gradients of sum(grad_out * S) for the transform; grad_out [(B,) n_dirs, K]. Returns
    grad_tau [K], grad_alpha, grad_u [n_dirs, ndim] and (want_img) grad_img, grad_img_absterms:
    the sums over directions of the single-direction gradients, with grad_u kept per direction."""
    nd = np.asarray(img).ndim if ndim is None else ndim
    U = _directions(U, nd)
    go = np.asarray(grad_out, np.float64)
    res = {"grad_tau": 0.0, "grad_alpha": 0.0, "grad_u": np.zeros(U.shape, np.float64)}
    if want_img:
        res["grad_img"] = 0.0
        res["grad_img_absterms"] = 0.0
    for j in range(U.shape[0]):
        r = ecc_soft_bwd(img, tau, lam, alpha, U[j], go[..., j, :], ndim=nd, want_img=want_img)
        res["grad_tau"] = res["grad_tau"] + r["grad_tau"]
        res["grad_alpha"] = res["grad_alpha"] + r["grad_alpha"]
        res["grad_u"][j] = r["grad_u"]
        if want_img:
            res["grad_img"] = res["grad_img"] + r["grad_img"]
            res["grad_img_absterms"] = res["grad_img_absterms"] + r["grad_img_absterms"]
    return res
