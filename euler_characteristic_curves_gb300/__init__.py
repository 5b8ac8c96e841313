"""Euler characteristic curves of dense 2-D/3-D grids on one GB300 (sm_103a).

The compute runs in the CUDA library built from ``csrc/`` behind the C ABI in
``include/ecc.h``; this package only marshals arguments (``ecc`` module). The native library is
loaded on first use and a missing library raises immediately: there is no CPU fallback.
"""
__all__ = ["ecc_hard", "ecc_hard_stream", "hard_stream_buffer_bytes", "ecc_soft_fwd",
           "ecc_soft_bwd", "ecc_soft_stats", "ecc_soft_fwd_noalloc", "soft_workspace_bytes",
           "SoftECC", "soft_ecc", "ecc_soft_ect_fwd", "ecc_soft_ect_bwd", "ecc_soft_ect_stats",
           "SoftECT", "soft_ect"]


def __getattr__(name):
    if name in __all__:
        from . import ecc

        return getattr(ecc, name)
    raise AttributeError(name)
