"""Thin Python binding of the C ABI in include/ecc.h (argument marshalling only).

Every computation runs in the CUDA library libecc_gb300.so; this module checks shapes, passes
device pointers, sizes and the current CUDA stream, and turns negative status codes into
exceptions. There is no CPU path: CPU tensors are rejected, and a missing library raises.

Names follow the C entry points: ``ecc_hard``, ``ecc_hard_partial``, ``hist_to_curve``,
``hard_launch_info``, ``device_status``, ``wait_probe``, ``ecc_hard_stream``, ``ecc_soft_fwd``, ``ecc_soft_bwd``,
``ecc_soft_stats``, ``ecc_soft_fwd_noalloc``, ``ecc_soft_ect_fwd``, ``ecc_soft_ect_bwd``,
``ecc_soft_ect_stats``, ``soft_workspace_bytes``; ``SoftECT`` / ``soft_ect`` wrap the transform; ``SoftECC`` / ``soft_ecc`` wrap the soft pair as a differentiable
PyTorch layer ("Key designs -- differentiable ECC layer (sigmoid relaxation)" in the paper notes
"Scalable GPU-Accelerated Euler Characteristic Curves").
"""
from __future__ import annotations

import contextlib
import ctypes
import functools
import os
import threading

import torch

from . import build as _build

ECC_U8, ECC_F32 = 0, 1
_lock = threading.Lock()
_lib = None


def debug_requested() -> bool:
    """ECC_DEBUG=1 selects the bounds-checked debug build of the library."""
    return os.environ.get("ECC_DEBUG", "") == "1"


def library_path() -> str:
    return _build.DEBUG_LIB_PATH if debug_requested() else _build.LIB_PATH


def load_library():
    """Load libecc_gb300.so (built in-tree by ``build.build()``), or its bounds-checked debug
    variant when ECC_DEBUG=1 (``build.build(debug=True)``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            flag = " --debug" if debug_requested() else ""
            raise RuntimeError(
                f"ECC CUDA library not found at {path}; build it first with "
                f"`python -m euler_characteristic_curves_gb300.build{flag}` (there is no CPU "
                "fallback)")
        lib = ctypes.CDLL(path)
        p, i, i64, d, f, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double,
                               ctypes.c_float, ctypes.c_size_t)
        lib.ecc_hard.argtypes = [p, i, i, p, i64, i, d, d, p, p]
        lib.ecc_hard.restype = i
        lib.ecc_hard_partial.argtypes = [p, i, i, p, i64, i, d, d, i, p, p]
        lib.ecc_hard_partial.restype = i
        lib.ecc_hist_to_curve.argtypes = [p, i, i64, p]
        lib.ecc_hist_to_curve.restype = i
        lib.ecc_device_status.argtypes = [i]
        lib.ecc_device_status.restype = i
        lib.ecc_device_error_bits.argtypes = [i]
        lib.ecc_device_error_bits.restype = i64
        lib.ecc_debug_build.argtypes = []
        lib.ecc_debug_build.restype = i
        lib.ecc_wait_probe.argtypes = [i64, p]
        lib.ecc_wait_probe.restype = i
        lib.ecc_hard_launch_info.argtypes = [i, i, p, i64, i, i, p]
        lib.ecc_hard_launch_info.restype = i
        lib.ecc_hard_stream_buffer_bytes.argtypes = [i, p, i]
        lib.ecc_hard_stream_buffer_bytes.restype = sz
        lib.ecc_hard_stream.argtypes = [p, i, p, i, d, d, i, p, sz, p, p]
        lib.ecc_hard_stream.restype = i
        lib.ecc_soft_workspace_bytes.argtypes = [i, p, i64, i]
        lib.ecc_soft_workspace_bytes.restype = sz
        lib.ecc_soft_fwd.argtypes = [p, i, p, i64, p, i, f, p, p, p, p, sz, p]
        lib.ecc_soft_fwd.restype = i
        lib.ecc_soft_bwd.argtypes = [p, i, p, i64, p, i, f, p, p, p, p, p, p, p, p, sz, p]
        lib.ecc_soft_bwd.restype = i
        lib.ecc_soft_ect_workspace_bytes.argtypes = [i, p, i64, i, i]
        lib.ecc_soft_ect_workspace_bytes.restype = sz
        lib.ecc_soft_ect_fwd.argtypes = [p, i, p, i64, p, i, f, p, p, i, p, p, sz, p]
        lib.ecc_soft_ect_fwd.restype = i
        lib.ecc_soft_ect_bwd.argtypes = [p, i, p, i64, p, i, f, p, p, i, p, p, p, p, p, p, sz, p]
        lib.ecc_soft_ect_bwd.restype = i
        lib.ecc_soft_ect_stats.argtypes = [i, p, i64, i, i, p, sz, p, p]
        lib.ecc_soft_ect_stats.restype = i
        lib.ecc_soft_stats.argtypes = [i, p, i64, i, p, sz, p, p]
        lib.ecc_soft_stats.restype = i
        lib.ecc_soft_fwd_noalloc.argtypes = [p, i, p, i64, p, i, f, p, p, p, p]
        lib.ecc_soft_fwd_noalloc.restype = i
        lib.ecc_status_str.argtypes = [i]
        lib.ecc_status_str.restype = ctypes.c_char_p
        lib.ecc_version.argtypes = []
        lib.ecc_version.restype = i
        _lib = lib
        return lib


class ECCError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = load_library().ecc_status_str(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")
        self.status = status


def _check(rc: int, where: str):
    if rc != 0:
        raise ECCError(rc, where)


@functools.lru_cache(maxsize=256)
def _dims_tuple_array(dims):
    return (ctypes.c_int64 * len(dims))(*dims)  # read-only for the library (const int64_t *)


def _dims_array(dims):
    return _dims_tuple_array(tuple(int(x) for x in dims))


# The current stream's raw handle without building a Stream object (a few microseconds per call
# on small inputs); the public call where this build of torch lacks it.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(stream):
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


_no_switch = contextlib.nullcontext()


def _on_device(t: torch.Tensor):
    """Makes t's device current for a library call: the library launches on the current device,
    and the current stream is looked up there. No switch when it already is current."""
    idx = t.device.index
    if idx is None or idx == torch.cuda.current_device():
        return _no_switch
    return torch.cuda.device(idx)


def _check_out(out: torch.Tensor, like: torch.Tensor, dtype, numel: int):
    """A caller-supplied output must be a contiguous tensor of `dtype` with `numel` elements on
    the input's device (the library writes exactly that many)."""
    _need_cuda(out, "out")
    if out.dtype != dtype or out.numel() != numel or out.device != like.device:
        raise ValueError(f"out must be {dtype} with {numel} elements on {like.device}")


def _need_cuda(t: torch.Tensor, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor (the ECC library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _split(img: torch.Tensor, ndim):
    if ndim is None:
        if img.dim() == 2:
            ndim = 2
        elif img.dim() == 4:
            ndim = 3
        else:
            raise ValueError("pass ndim=2 (batch of images) or ndim=3 (one volume) for a 3-D "
                             "tensor")
    if img.dim() == ndim:
        return ndim, 1, tuple(img.shape), False
    if img.dim() == ndim + 1:
        return ndim, img.shape[0], tuple(img.shape[1:]), True
    raise ValueError(f"tensor of shape {tuple(img.shape)} is not a {ndim}-D image or a batch")


def ecc_hard(img: torch.Tensor, nbins: int, vmin: float, vmax: float, ndim: int | None = None,
             out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Hard ECC: int64 [batch, nbins] (or [nbins] for one unbatched image) on img's device.

    img: uint8 or float32 CUDA tensor [(B,) (D,) H, W]. Thresholds t_k are nbins uniform values
    from vmin to vmax inclusive; out[b, k] = ECC of image b at t_k.
    """
    _need_cuda(img, "img")
    if img.dtype == torch.uint8:
        dt = ECC_U8
    elif img.dtype == torch.float32:
        dt = ECC_F32
    else:
        raise TypeError(f"img dtype {img.dtype}: uint8 or float32 expected")
    ndim, batch, dims, batched = _split(img, ndim)
    if out is None:
        out = torch.empty((batch, nbins), dtype=torch.int64, device=img.device)
    else:
        _check_out(out, img, torch.int64, batch * nbins)
    lib = load_library()
    with _on_device(img):
        rc = lib.ecc_hard(img.data_ptr(), dt, ndim, _dims_array(dims), batch, int(nbins),
                          float(vmin), float(vmax), out.data_ptr(), _stream_handle(stream))
    _check(rc, "ecc_hard")
    out = out.view(batch, nbins)
    return out if batched else out[0]


def ecc_hard_partial(img: torch.Tensor, nbins: int, vmin: float, vmax: float, hist: torch.Tensor,
                     sign: int = 1, ndim: int | None = None, stream=None) -> torch.Tensor:
    """Adds sign * (the unscanned per-bin cell counts of img) into hist (int64 [batch, nbins] on
    img's device, not zeroed): the partial that sharded calls sum before one running sum
    (``hist_to_curve``). img as for ``ecc_hard``."""
    _need_cuda(img, "img")
    if img.dtype == torch.uint8:
        dt = ECC_U8
    elif img.dtype == torch.float32:
        dt = ECC_F32
    else:
        raise TypeError(f"img dtype {img.dtype}: uint8 or float32 expected")
    ndim, batch, dims, _ = _split(img, ndim)
    _check_out(hist, img, torch.int64, batch * nbins)
    with _on_device(img):
        rc = load_library().ecc_hard_partial(img.data_ptr(), dt, ndim, _dims_array(dims), batch,
                                             int(nbins), float(vmin), float(vmax), int(sign),
                                             hist.data_ptr(), _stream_handle(stream))
    _check(rc, "ecc_hard_partial")
    return hist


def hist_to_curve(hist: torch.Tensor, stream=None) -> torch.Tensor:
    """In place: hist[..., k] becomes the running sum over bins 0..k (int64 CUDA tensor, last axis
    the bins). Returns hist."""
    _need_cuda(hist, "hist")
    if hist.dtype != torch.int64 or hist.dim() < 1:
        raise ValueError("hist must be an int64 tensor with the bins on its last axis")
    nbins = hist.shape[-1]
    with _on_device(hist):
        rc = load_library().ecc_hist_to_curve(hist.data_ptr(), int(nbins),
                                              hist.numel() // max(1, nbins),
                                              _stream_handle(stream))
    _check(rc, "ecc_hist_to_curve")
    return hist


def device_error_bits(clear: bool = True, device=None) -> int:
    """ecc_device_error_bits on ``device`` (default: the current one): the raw error-word bits
    (bit 0 a wait gave up; the others debug-build bounds checks, see include/ecc.h)."""
    ctx = torch.cuda.device(device) if device is not None else _no_switch
    with ctx:
        return int(load_library().ecc_device_error_bits(1 if clear else 0))


def device_status(clear: bool = True, device=None) -> int:
    """ecc_device_status on ``device`` (default: the current one): 0, or the ECC_ETIMEOUT status
    when a kernel gave up waiting for its own staged copy since the last clear."""
    ctx = torch.cuda.device(device) if device is not None else _no_switch
    with ctx:
        return int(load_library().ecc_device_status(1 if clear else 0))


def wait_probe(limit_ns: int, device=None, stream=None) -> None:
    """ecc_wait_probe on ``device`` (default: the current one): a kernel that waits, with the
    kernels' bounded wait cut to ``limit_ns``, for an mbarrier nothing completes, then records a
    wait timeout in the device error word (read it with ``device_status``)."""
    ctx = torch.cuda.device(device) if device is not None else _no_switch
    with ctx:
        _check(load_library().ecc_wait_probe(int(limit_ns), _stream_handle(stream)),
               "ecc_wait_probe")


def hard_launch_info(dims, batch: int, nbins: int, dtype=torch.float32, sm_count: int = 0):
    """The launch shape ecc_hard takes for these sizes (ecc_hard_launch_info): a dict with
    blocks_per_image, tasks_per_image, rows_per_task, rounds, direct and sms. ``sm_count`` 0
    plans for the current device."""
    dt = ECC_U8 if dtype == torch.uint8 else ECC_F32
    info = (ctypes.c_int64 * 6)()
    _check(load_library().ecc_hard_launch_info(dt, len(dims), _dims_array(dims), int(batch),
                                               int(nbins), int(sm_count), info),
           "ecc_hard_launch_info")
    keys = ("blocks_per_image", "tasks_per_image", "rows_per_task", "rounds", "direct", "sms")
    return dict(zip(keys, (int(v) for v in info)))


def hard_stream_buffer_bytes(dims, dtype, slab_planes: int) -> int:
    """Device bytes that ecc_hard_stream needs for a [D, H, W] volume of this dtype."""
    dt = ECC_U8 if dtype == torch.uint8 else ECC_F32
    return int(load_library().ecc_hard_stream_buffer_bytes(dt, _dims_array(dims),
                                                           int(slab_planes)))


def ecc_hard_stream(img: torch.Tensor, nbins: int, vmin: float, vmax: float,
                    slab_planes: int = 64, buf: torch.Tensor | None = None,
                    out: torch.Tensor | None = None, device=None, stream=None) -> torch.Tensor:
    """Hard ECC of one [D, H, W] volume that need not fit on the device: the volume (a CPU
    tensor, page-locked for overlapped copies, or a CUDA tensor) is streamed through two slab
    buffers of `slab_planes` planes. Returns int64 [nbins] on `device` (default cuda:0)."""
    if not isinstance(img, torch.Tensor) or img.dim() != 3 or not img.is_contiguous():
        raise ValueError("img must be a contiguous [D, H, W] tensor")
    if img.dtype == torch.uint8:
        dt = ECC_U8
    elif img.dtype == torch.float32:
        dt = ECC_F32
    else:
        raise TypeError(f"img dtype {img.dtype}: uint8 or float32 expected")
    dev = torch.device(device) if device is not None else (
        img.device if img.is_cuda else torch.device("cuda", 0))
    if dev.type != "cuda":
        raise TypeError("the streamed ECC runs on a CUDA device (there is no CPU path)")
    dims = tuple(img.shape)
    need = hard_stream_buffer_bytes(dims, img.dtype, slab_planes)
    if need == 0:
        raise ValueError("unsupported sizes for the streamed ECC")
    if buf is None:
        buf = torch.empty(need, dtype=torch.uint8, device=dev)
    elif not buf.is_cuda or buf.numel() < need:
        raise ValueError(f"buf must be a CUDA tensor of at least {need} bytes")
    if out is None:
        out = torch.empty(nbins, dtype=torch.int64, device=dev)
    elif (not out.is_cuda or not out.is_contiguous() or out.dtype != torch.int64
          or out.numel() != nbins or out.device != buf.device):
        raise ValueError(f"out must be a contiguous int64 CUDA tensor of {nbins} elements on "
                         f"{buf.device}")
    with torch.cuda.device(dev):
        rc = load_library().ecc_hard_stream(ctypes.c_void_p(img.data_ptr()), dt,
                                            _dims_array(dims), int(nbins), float(vmin),
                                            float(vmax), int(slab_planes),
                                            ctypes.c_void_p(buf.data_ptr()), buf.numel(),
                                            ctypes.c_void_p(out.data_ptr()),
                                            _stream_handle(stream))
    _check(rc, "ecc_hard_stream")
    return out


def soft_workspace_bytes(dims, batch: int, K: int, ndirs: int = 1) -> int:
    lib = load_library()
    return int(lib.ecc_soft_ect_workspace_bytes(len(dims), _dims_array(dims), int(batch), int(K),
                                                int(ndirs)))


def _soft_common(img, tau, alpha, u, ndim):
    _need_cuda(img, "img")
    if img.dtype != torch.float32:
        raise TypeError("soft ECC takes float32 images")
    for name, t in (("tau", tau), ("alpha", alpha), ("u", u)):
        _need_cuda(t, name)
        if t.dtype != torch.float32:
            raise TypeError(f"{name} must be float32")
    ndim = u.numel() if ndim is None else ndim  # u has one component per image axis
    ndim, batch, dims, batched = _split(img, ndim)
    if alpha.numel() != 1 or u.numel() != ndim:
        raise ValueError(f"alpha must have 1 element and u {ndim}")
    return ndim, batch, dims, batched


def _workspace(ws, dims, batch, K, device, ndirs=1):
    need = soft_workspace_bytes(dims, batch, K, ndirs)
    if need == 0:
        raise ValueError("unsupported soft-ECC sizes")
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=device)
    elif ws.numel() < need:
        raise ValueError(f"workspace of {ws.numel()} bytes, {need} needed")
    return ws


def ecc_soft_fwd(img, tau, lam: float, alpha, u, ws=None, out=None, ndim=None, stream=None):
    """Soft ECC S[b, k] (float32). Returns (S, ws); pass ws unchanged to ecc_soft_bwd."""
    ndim, batch, dims, batched = _soft_common(img, tau, alpha, u, ndim)
    K = tau.numel()
    ws = _workspace(ws, dims, batch, K, img.device)
    if out is None:
        out = torch.empty((batch, K), dtype=torch.float32, device=img.device)
    else:
        _check_out(out, img, torch.float32, batch * K)
    lib = load_library()
    with _on_device(img):
        rc = lib.ecc_soft_fwd(ctypes.c_void_p(img.data_ptr()), ndim, _dims_array(dims), batch,
                              ctypes.c_void_p(tau.data_ptr()), K, float(lam),
                              ctypes.c_void_p(alpha.data_ptr()), ctypes.c_void_p(u.data_ptr()),
                              ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(ws.data_ptr()),
                              ws.numel(), _stream_handle(stream))
    _check(rc, "ecc_soft_fwd")
    out = out.view(batch, K)
    return (out if batched else out[0]), ws


def ecc_soft_stats(img, K: int, ws, ndim=None, stream=None) -> torch.Tensor:
    """int64 CUDA tensor [3]: voxels on the soft work list (summed over the batch), tiles that
    took the direct exponent form, and tiles, for the workspace ``ws`` that a soft forward call
    filled for ``img`` and ``K`` thresholds (``ndim``: 2 or 3, default 2 for [B, H, W])."""
    _need_cuda(img, "img")
    _need_cuda(ws, "ws")
    ndim, batch, dims, _ = _split(img, 2 if ndim is None and img.dim() != 4 else ndim)
    stats = torch.empty(3, dtype=torch.int64, device=img.device)
    with _on_device(img):
        rc = load_library().ecc_soft_stats(ndim, _dims_array(dims), batch, int(K),
                                           ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                           ctypes.c_void_p(stats.data_ptr()),
                                           _stream_handle(stream))
    _check(rc, "ecc_soft_stats")
    return stats


def ecc_soft_fwd_noalloc(img, tau, lam: float, alpha, u, out=None, ndim=None, stream=None):
    """Soft ECC S[b, k] of 2-D images through ecc_soft_fwd_noalloc: same result as
    ecc_soft_fwd, but the workspace is the library's own fixed device array, so the call
    allocates no device memory (``out`` may be passed pre-allocated too). Volumes and sizes
    needing more than the array raise."""
    ndim, batch, dims, batched = _soft_common(img, tau, alpha, u, ndim)
    K = tau.numel()
    if out is None:
        out = torch.empty((batch, K), dtype=torch.float32, device=img.device)
    else:
        _check_out(out, img, torch.float32, batch * K)
    lib = load_library()
    with _on_device(img):
        rc = lib.ecc_soft_fwd_noalloc(ctypes.c_void_p(img.data_ptr()), ndim, _dims_array(dims),
                                      batch, ctypes.c_void_p(tau.data_ptr()), K, float(lam),
                                      ctypes.c_void_p(alpha.data_ptr()),
                                      ctypes.c_void_p(u.data_ptr()),
                                      ctypes.c_void_p(out.data_ptr()), _stream_handle(stream))
    _check(rc, "ecc_soft_fwd_noalloc")
    out = out.view(batch, K)
    return out if batched else out[0]


def ecc_soft_bwd(img, tau, lam: float, alpha, u, grad_out, ws, want_img: bool = False, ndim=None,
                 stream=None):
    """Analytic gradients of sum(grad_out * S): dict of float32 CUDA tensors grad_tau [K],
    grad_alpha [1], grad_u [ndim] and, when want_img, grad_img (img's shape)."""
    ndim, batch, dims, batched = _soft_common(img, tau, alpha, u, ndim)
    K = tau.numel()
    _need_cuda(grad_out, "grad_out")
    if grad_out.dtype != torch.float32 or grad_out.numel() != batch * K:
        raise ValueError("grad_out must be float32 with batch * K elements")
    ws = _workspace(ws, dims, batch, K, img.device)
    dev = img.device
    gt = torch.empty(K, dtype=torch.float32, device=dev)
    ga = torch.empty(1, dtype=torch.float32, device=dev)
    gu = torch.empty(ndim, dtype=torch.float32, device=dev)
    gi = torch.empty_like(img) if want_img else None
    lib = load_library()
    with _on_device(img):
        rc = lib.ecc_soft_bwd(ctypes.c_void_p(img.data_ptr()), ndim, _dims_array(dims), batch,
                              ctypes.c_void_p(tau.data_ptr()), K, float(lam),
                              ctypes.c_void_p(alpha.data_ptr()), ctypes.c_void_p(u.data_ptr()),
                              ctypes.c_void_p(grad_out.data_ptr()),
                              ctypes.c_void_p(gt.data_ptr()), ctypes.c_void_p(ga.data_ptr()),
                              ctypes.c_void_p(gu.data_ptr()),
                              ctypes.c_void_p(gi.data_ptr() if gi is not None else None),
                              ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream_handle(stream))
    _check(rc, "ecc_soft_bwd")
    res = {"grad_tau": gt, "grad_alpha": ga, "grad_u": gu}
    if want_img:
        res["grad_img"] = gi
    return res


def _ect_common(img, tau, alpha, U, ndim):
    _need_cuda(U, "u")
    if U.dim() != 2:
        raise ValueError("directions must have shape [n_dirs, ndim]")
    ndim = U.shape[1] if ndim is None else ndim
    if U.shape[1] != ndim:
        raise ValueError(f"directions must have {ndim} components")
    for name, t in (("tau", tau), ("alpha", alpha)):
        _need_cuda(t, name)
        if t.dtype != torch.float32:
            raise TypeError(f"{name} must be float32")
    if U.dtype != torch.float32:
        raise TypeError("u must be float32")
    _need_cuda(img, "img")
    if img.dtype != torch.float32:
        raise TypeError("soft ECC takes float32 images")
    if alpha.numel() != 1:
        raise ValueError("alpha must have 1 element")
    ndim, batch, dims, batched = _split(img, ndim)
    return ndim, batch, dims, batched, U.shape[0]


def ecc_soft_ect_fwd(img, tau, lam: float, alpha, U, ws=None, out=None, ndim=None, stream=None):
    """Soft Euler characteristic transform S[b, j, k]: the soft ECC of image b along direction
    U[j] (U: float32 CUDA [n_dirs, ndim]). Returns (S, ws); pass ws unchanged to the backward."""
    ndim, batch, dims, batched, nd = _ect_common(img, tau, alpha, U, ndim)
    K = tau.numel()
    ws = _workspace(ws, dims, batch, K, img.device, nd)
    if out is None:
        out = torch.empty((batch, nd, K), dtype=torch.float32, device=img.device)
    else:
        _check_out(out, img, torch.float32, batch * nd * K)
    lib = load_library()
    with _on_device(img):
        rc = lib.ecc_soft_ect_fwd(ctypes.c_void_p(img.data_ptr()), ndim, _dims_array(dims),
                                  batch, ctypes.c_void_p(tau.data_ptr()), K, float(lam),
                                  ctypes.c_void_p(alpha.data_ptr()),
                                  ctypes.c_void_p(U.data_ptr()), nd,
                                  ctypes.c_void_p(out.data_ptr()),
                                  ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                  _stream_handle(stream))
    _check(rc, "ecc_soft_ect_fwd")
    out = out.view(batch, nd, K)
    return (out if batched else out[0]), ws


def ecc_soft_ect_bwd(img, tau, lam: float, alpha, U, grad_out, ws, want_img: bool = False,
                     ndim=None, stream=None):
    """Gradients of sum(grad_out * S) for the transform: grad_tau [K], grad_alpha [1],
    grad_u [n_dirs, ndim] and, when want_img, grad_img (summed over directions)."""
    ndim, batch, dims, batched, nd = _ect_common(img, tau, alpha, U, ndim)
    K = tau.numel()
    _need_cuda(grad_out, "grad_out")
    if grad_out.dtype != torch.float32 or grad_out.numel() != batch * nd * K:
        raise ValueError("grad_out must be float32 with batch * n_dirs * K elements")
    ws = _workspace(ws, dims, batch, K, img.device, nd)
    dev = img.device
    gt = torch.empty(K, dtype=torch.float32, device=dev)
    ga = torch.empty(1, dtype=torch.float32, device=dev)
    gu = torch.empty((nd, ndim), dtype=torch.float32, device=dev)
    gi = torch.empty_like(img) if want_img else None
    lib = load_library()
    with _on_device(img):
        rc = lib.ecc_soft_ect_bwd(ctypes.c_void_p(img.data_ptr()), ndim, _dims_array(dims),
                                  batch, ctypes.c_void_p(tau.data_ptr()), K, float(lam),
                                  ctypes.c_void_p(alpha.data_ptr()),
                                  ctypes.c_void_p(U.data_ptr()), nd,
                                  ctypes.c_void_p(grad_out.data_ptr()),
                                  ctypes.c_void_p(gt.data_ptr()), ctypes.c_void_p(ga.data_ptr()),
                                  ctypes.c_void_p(gu.data_ptr()),
                                  ctypes.c_void_p(gi.data_ptr() if gi is not None else None),
                                  ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                  _stream_handle(stream))
    _check(rc, "ecc_soft_ect_bwd")
    res = {"grad_tau": gt, "grad_alpha": ga, "grad_u": gu}
    if want_img:
        res["grad_img"] = gi
    return res


def ecc_soft_ect_stats(img, K: int, ndirs: int, ws, ndim=None, stream=None) -> torch.Tensor:
    """ecc_soft_stats for a workspace filled by ecc_soft_ect_fwd."""
    _need_cuda(img, "img")
    _need_cuda(ws, "ws")
    ndim, batch, dims, _ = _split(img, 2 if ndim is None and img.dim() != 4 else ndim)
    stats = torch.empty(3, dtype=torch.int64, device=img.device)
    with _on_device(img):
        rc = load_library().ecc_soft_ect_stats(ndim, _dims_array(dims), batch, int(K),
                                               int(ndirs), ctypes.c_void_p(ws.data_ptr()),
                                               ws.numel(), ctypes.c_void_p(stats.data_ptr()),
                                               _stream_handle(stream))
    _check(rc, "ecc_soft_ect_stats")
    return stats


class SoftECT(torch.autograd.Function):
    """Differentiable soft Euler characteristic transform: S = SoftECT.apply(img, tau, alpha, U, lam).

    img float32 [(B,) H, W] or [(B,) D, H, W]; U [n_dirs, ndim] directions; tau [K]; alpha [1];
    returns [(B,) n_dirs, K]. Gradients flow to tau, alpha, U and, when it requires grad, img.
    """

    @staticmethod
    def forward(ctx, img, tau, alpha, U, lam):
        img, tau, alpha, U = (t.contiguous() for t in (img, tau, alpha, U))
        out, ws = ecc_soft_ect_fwd(img, tau, lam, alpha, U)
        ctx.save_for_backward(img, tau, alpha, U, ws)
        ctx.lam = float(lam)
        return out

    @staticmethod
    def backward(ctx, grad_out):
        img, tau, alpha, U, ws = ctx.saved_tensors
        res = ecc_soft_ect_bwd(img, tau, ctx.lam, alpha, U, grad_out.contiguous().float(), ws,
                               want_img=ctx.needs_input_grad[0])
        gi = res.get("grad_img")
        return (gi, res["grad_tau"], res["grad_alpha"].view_as(alpha), res["grad_u"].view_as(U),
                None)


def soft_ect(img, tau, alpha, U, lam: float):
    return SoftECT.apply(img, tau, alpha, U, lam)


class SoftECC(torch.autograd.Function):
    """Differentiable soft ECC layer: S = SoftECC.apply(img, tau, alpha, u, lam).

    img float32 [(B,) H, W] with u [2], or [(B,) D, H, W] with u [3]; tau [K]; alpha [1]
    (tau, alpha and u learnable); lam a Python float.
    Gradients flow to tau, alpha, u and, when it requires grad, img.
    """

    @staticmethod
    def forward(ctx, img, tau, alpha, u, lam):
        img, tau, alpha, u = (t.contiguous() for t in (img, tau, alpha, u))
        out, ws = ecc_soft_fwd(img, tau, lam, alpha, u)
        ctx.save_for_backward(img, tau, alpha, u, ws)
        ctx.lam = float(lam)
        return out

    @staticmethod
    def backward(ctx, grad_out):
        img, tau, alpha, u, ws = ctx.saved_tensors
        res = ecc_soft_bwd(img, tau, ctx.lam, alpha, u, grad_out.contiguous().float(), ws,
                           want_img=ctx.needs_input_grad[0])
        gi = res.get("grad_img")
        return (gi, res["grad_tau"], res["grad_alpha"].view_as(alpha), res["grad_u"].view_as(u),
                None)


def soft_ecc(img, tau, alpha, u, lam: float):
    return SoftECC.apply(img, tau, alpha, u, lam)
