"""The C-ABI library on a machine without a GPU: it loads, exports every function that
include/ecc.h declares, and its host-side validation returns the documented status codes before
any CUDA call (no compute call is made here)."""
import ctypes
import os
import re

import pytest

from euler_characteristic_curves_gb300 import build as libbuild
from euler_characteristic_curves_gb300 import ecc

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "ecc.h")
OK, EINVAL, EDTYPE, EDIM, EWS, ECUDA, ERANGE = 0, -1, -2, -3, -4, -5, -6


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return ecc.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ecc_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"ecc_hard", "ecc_soft_fwd", "ecc_soft_bwd", "ecc_soft_workspace_bytes",
            "ecc_status_str", "ecc_version"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_wait_probe_validation(lib):
    """The wait-timeout probe rejects limits outside (0, 2 s] before it touches a device."""
    lib.ecc_wait_probe.argtypes = [ctypes.c_int64, ctypes.c_void_p]
    assert lib.ecc_wait_probe(0, None) == EINVAL
    assert lib.ecc_wait_probe(-5, None) == EINVAL
    assert lib.ecc_wait_probe(2_000_000_001, None) == ERANGE


def test_status_strings_and_version(lib):
    for code in (OK, EINVAL, EDTYPE, EDIM, EWS, ECUDA, ERANGE, 12345):
        s = lib.ecc_status_str(code)
        assert isinstance(s, bytes) and len(s) > 0
    assert lib.ecc_status_str(EWS).startswith(b"ECC_EWS")
    assert lib.ecc_version() >= 10000


def dims(*v):
    return (ctypes.c_int64 * len(v))(*v)


FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first


def test_hard_validation(lib):
    d2 = dims(8, 8)
    h = lib.ecc_hard
    assert h(None, 1, 2, d2, 1, 4, 0.0, 1.0, FAKE, None) == EINVAL
    assert h(FAKE, 1, 2, d2, 1, 4, 0.0, 1.0, None, None) == EINVAL
    assert h(FAKE, 1, 2, None, 1, 4, 0.0, 1.0, FAKE, None) == EINVAL
    assert h(FAKE, 7, 2, d2, 1, 4, 0.0, 1.0, FAKE, None) == EDTYPE
    assert h(FAKE, 1, 1, d2, 1, 4, 0.0, 1.0, FAKE, None) == EDIM
    assert h(FAKE, 1, 4, dims(2, 2, 2, 2), 1, 4, 0.0, 1.0, FAKE, None) == EDIM
    assert h(FAKE, 1, 2, dims(0, 8), 1, 4, 0.0, 1.0, FAKE, None) == EDIM
    assert h(FAKE, 1, 2, d2, 0, 4, 0.0, 1.0, FAKE, None) == EINVAL
    assert h(FAKE, 1, 2, d2, 1, 0, 0.0, 1.0, FAKE, None) == EINVAL
    assert h(FAKE, 1, 2, d2, 1, 4097, 0.0, 1.0, FAKE, None) == ERANGE
    assert h(FAKE, 1, 2, d2, 1, 4, 1.0, 0.0, FAKE, None) == EINVAL
    assert h(FAKE, 1, 2, d2, 1, 4, float("nan"), 1.0, FAKE, None) == EINVAL
    assert h(FAKE, 1, 2, d2, 1, 4, 0.0, float("inf"), FAKE, None) == EINVAL
    assert h(FAKE, 1, 2, d2, 1, 4, -1.7e308, 1.7e308, FAKE, None) == EINVAL
    assert h(FAKE, 1, 2, dims(1 << 40, 1 << 30), 1, 4, 0.0, 1.0, FAKE, None) == ERANGE


MAX_EXTENT = 1 << 30  # ECC_MAX_EXTENT


def test_extents_the_kernels_cannot_index_are_rejected(lib):
    """Every axis is limited to ECC_MAX_EXTENT: the kernels index rows, columns and strips with
    32-bit integers, so a longer axis returns ECC_ERANGE before any launch instead of wrapping.
    The pointers are fakes that are never dereferenced."""
    h = lib.ecc_hard
    for dt in (0, 1):
        assert h(FAKE, dt, 2, dims(1, 3 * 10**9), 1, 4, 0.0, 1.0, FAKE, None) == ERANGE
        assert h(FAKE, dt, 2, dims(3 * 10**9, 1), 1, 4, 0.0, 1.0, FAKE, None) == ERANGE
        assert h(FAKE, dt, 2, dims(1, MAX_EXTENT + 1), 1, 4, 0.0, 1.0, FAKE, None) == ERANGE
        assert h(FAKE, dt, 3, dims(1, 1, 3 * 10**9), 1, 4, 0.0, 1.0, FAKE, None) == ERANGE
        assert h(FAKE, dt, 3, dims(3 * 10**9, 1, 1), 1, 4, 0.0, 1.0, FAKE, None) == ERANGE
        assert h(FAKE, dt, 3, dims(1, MAX_EXTENT + 1, 1), 1, 4, 0.0, 1.0, FAKE, None) == ERANGE
        # 2-D: one warp per (128-column strip, row range), at most 2^31 of them
        assert h(FAKE, dt, 2, dims(MAX_EXTENT, 300), 1, 4, 0.0, 1.0, FAKE, None) == ERANGE
    bb = lib.ecc_hard_stream_buffer_bytes
    assert bb(1, dims(4, 1, 3 * 10**9), 2) == 0
    assert bb(1, dims(4, MAX_EXTENT + 1, 1), 2) == 0
    st = lib.ecc_hard_stream
    buf = ctypes.c_void_p(0x100000)
    assert st(FAKE, 1, dims(4, 1, 3 * 10**9), 8, 0.0, 1.0, 2, buf, 1 << 40, FAKE, None) == ERANGE
    w = lib.ecc_soft_workspace_bytes
    assert w(2, dims(1, MAX_EXTENT + 1), 1, 4) == 0
    assert w(3, dims(MAX_EXTENT + 1, 1, 1), 1, 4) == 0
    f = lib.ecc_soft_fwd
    ws = ctypes.c_void_p(0x100000)
    assert f(FAKE, 2, dims(1, 3 * 10**9), 1, FAKE, 8, 50.0, FAKE, FAKE, FAKE, ws, 1 << 40,
             None) == ERANGE


def test_partial_and_curve_validation(lib):
    p = lib.ecc_hard_partial
    d2 = dims(8, 8)
    assert p(None, 1, 2, d2, 1, 4, 0.0, 1.0, 1, FAKE, None) == EINVAL
    assert p(FAKE, 1, 2, d2, 1, 4, 0.0, 1.0, 1, None, None) == EINVAL
    assert p(FAKE, 1, 2, d2, 1, 4, 0.0, 1.0, 0, FAKE, None) == EINVAL  # sign must be +1 / -1
    assert p(FAKE, 1, 2, d2, 1, 4, 0.0, 1.0, 2, FAKE, None) == EINVAL
    assert p(FAKE, 9, 2, d2, 1, 4, 0.0, 1.0, 1, FAKE, None) == EDTYPE
    assert p(FAKE, 1, 5, d2, 1, 4, 0.0, 1.0, -1, FAKE, None) == EDIM
    assert p(FAKE, 1, 2, d2, 1, 4097, 0.0, 1.0, 1, FAKE, None) == ERANGE
    assert p(FAKE, 1, 2, d2, 1, 4, 1.0, 0.0, 1, FAKE, None) == EINVAL
    assert p(FAKE, 1, 2, dims(1, 3 * 10**9), 1, 4, 0.0, 1.0, 1, FAKE, None) == ERANGE
    c = lib.ecc_hist_to_curve
    assert c(None, 4, 1, None) == EINVAL
    assert c(FAKE, 0, 1, None) == EINVAL and c(FAKE, 4, 0, None) == EINVAL
    assert c(FAKE, 4097, 1, None) == ERANGE and c(FAKE, 4, 65536, None) == ERANGE


def test_launch_info(lib):
    info = (ctypes.c_int64 * 6)()
    li = lib.ecc_hard_launch_info
    assert li(1, 3, dims(1024, 1024, 1024), 1, 256, 152, info) == OK
    blocks, tasks, rows, rounds, direct, sms = list(info)
    # float32, rows of 4k values, <= 256 bins: the TMA-staged kernel's segments, each block a
    # contiguous share of the 8 x 32 tiles x 1024 planes, cut where a tile ends
    assert sms == 152 and blocks == 152 * 3 and rows == -(-(8 * 32 * 1024) // blocks)
    assert rounds == 2 and blocks < tasks < 2 * blocks
    assert li(0, 3, dims(1024, 1024, 1024), 1, 256, 152, info) == OK  # uint8: task rounds
    blocks, tasks, rows, rounds, direct, sms = list(info)
    assert rounds == -(-tasks // blocks) > 1 and tasks % (8 * 32) == 0
    assert li(1, 2, dims(128, 128), 1, 256, 152, info) == OK and info[4] == 1  # one block
    assert li(1, 2, dims(8192, 8192), 1, 1024, 152, info) == OK and info[4] == 0
    assert li(1, 3, dims(8, 8, 8), 1, 4097, 152, info) == ERANGE
    assert li(1, 3, dims(8, 8, 8), 1, 16, 152, None) == EINVAL


def test_soft_workspace_size(lib):
    w = lib.ecc_soft_workspace_bytes
    assert w(2, dims(256, 256), 64, 128) > 64 * 256 * 256 * 16
    assert w(2, dims(256, 256), 64, 128) % 256 == 0
    assert w(2, dims(256, 256), 64, 256) > w(2, dims(256, 256), 64, 128)
    assert w(3, dims(8, 8, 8), 1, 4) > 8 * 8 * 8 * 16
    assert w(4, dims(2, 2, 2, 2), 1, 4) == 0
    assert w(2, dims(8, 8), 65536, 4) == 0  # images run along a 16-bit grid axis
    assert w(2, dims(0, 8), 1, 4) == 0
    assert w(2, dims(8, 8), 0, 4) == 0
    assert w(2, dims(8, 8), 1, 0) == 0
    assert w(2, dims(8, 8), 1, 8193) == 0


def test_soft_validation(lib):
    d2 = dims(16, 16)
    need = lib.ecc_soft_workspace_bytes(2, d2, 1, 8)
    ws = ctypes.c_void_p(0x100000)  # 256-byte aligned fake address
    f = lib.ecc_soft_fwd
    args = [FAKE, 2, d2, 1, FAKE, 8, 50.0, FAKE, FAKE, FAKE, ws, need, None]

    def call(**over):
        a = list(args)
        names = ["img", "ndim", "dims", "batch", "tau", "K", "lam", "alpha", "u", "out", "ws",
                 "ws_bytes", "stream"]
        for k, v in over.items():
            a[names.index(k)] = v
        return f(*a)

    assert call(img=None) == EINVAL
    assert call(tau=None) == EINVAL
    assert call(alpha=None) == EINVAL
    assert call(u=None) == EINVAL
    assert call(out=None) == EINVAL
    assert call(ndim=4, dims=dims(4, 4, 4, 4)) == EDIM
    assert call(ndim=1, dims=dims(4)) == EDIM
    assert call(ndim=3, dims=dims(4, 0, 4)) == EDIM
    assert call(ndim=3, dims=dims(40, 40, 40)) == EWS  # 3-D volumes need their own size
    assert call(K=0) == EINVAL
    assert call(K=8193) == ERANGE
    assert call(lam=0.0) == EINVAL
    assert call(lam=float("nan")) == EINVAL
    assert call(ws=None) == EWS
    assert call(ws_bytes=need - 1) == EWS
    assert call(ws=ctypes.c_void_p(0x100010)) == EWS  # misaligned
    b = lib.ecc_soft_bwd
    assert b(FAKE, 2, d2, 1, FAKE, 8, 50.0, FAKE, FAKE, None, FAKE, FAKE, FAKE, None, ws, need,
             None) == EINVAL
    assert b(FAKE, 2, d2, 1, FAKE, 8, 50.0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, need,
             None) == EWS


def test_soft_stats_validation(lib):
    d2 = dims(16, 16)
    need = lib.ecc_soft_workspace_bytes(2, d2, 1, 8)
    ws = ctypes.c_void_p(0x100000)
    st = lib.ecc_soft_stats
    assert st(2, d2, 1, 8, ws, need, None, None) == EINVAL
    assert st(2, None, 1, 8, ws, need, FAKE, None) == EINVAL
    assert st(5, d2, 1, 8, ws, need, FAKE, None) == EDIM
    assert st(2, d2, 0, 8, ws, need, FAKE, None) == EINVAL
    assert st(2, d2, 1, 8, None, need, FAKE, None) == EWS
    assert st(2, d2, 1, 8, ws, need - 1, FAKE, None) == EWS
    assert st(2, d2, 1, 8, ctypes.c_void_p(0x100008), need, FAKE, None) == EWS


def test_ect_validation(lib):
    d2 = dims(16, 16)
    w = lib.ecc_soft_ect_workspace_bytes
    assert w(2, d2, 1, 8, 1) == lib.ecc_soft_workspace_bytes(2, d2, 1, 8)
    assert w(2, d2, 1, 8, 4) > w(2, d2, 1, 8, 1)
    assert w(2, d2, 1, 8, 0) == 0
    assert w(2, d2, 1, 8, 4097) == 0
    assert w(2, d2, 300, 8, 300) == 0  # batch * directions above 65535
    need = w(2, d2, 1, 8, 4)
    ws = ctypes.c_void_p(0x100000)
    f = lib.ecc_soft_ect_fwd
    assert f(FAKE, 2, d2, 1, FAKE, 8, 50.0, FAKE, FAKE, 0, FAKE, ws, need, None) == EINVAL
    assert f(FAKE, 2, d2, 1, FAKE, 8, 50.0, FAKE, FAKE, 4097, FAKE, ws, need, None) == ERANGE
    assert f(FAKE, 2, d2, 1, FAKE, 8, 50.0, FAKE, None, 4, FAKE, ws, need, None) == EINVAL
    assert f(FAKE, 2, d2, 1, FAKE, 8, 50.0, FAKE, FAKE, 4, FAKE, ws, need - 1, None) == EWS
    b = lib.ecc_soft_ect_bwd
    assert b(FAKE, 2, d2, 1, FAKE, 8, 50.0, FAKE, FAKE, 4, None, FAKE, FAKE, FAKE, None, ws,
             need, None) == EINVAL


def test_stream_validation(lib):
    d3 = dims(10, 16, 16)
    bb = lib.ecc_hard_stream_buffer_bytes
    assert bb(1, d3, 4) == 2 * 4 * 16 * 16 * 4  # two buffers of four f32 planes (256-aligned)
    assert bb(0, d3, 4) == 2 * 1024  # u8: 4 * 16 * 16 bytes, rounded to 256, twice
    assert bb(1, d3, 64) == 2 * 10 * 16 * 16 * 4  # at most the whole volume
    assert bb(1, d3, 1) == 0 and bb(7, d3, 4) == 0 and bb(1, dims(0, 4, 4), 4) == 0
    need = bb(1, d3, 4)
    buf = ctypes.c_void_p(0x100000)
    st = lib.ecc_hard_stream
    assert st(None, 1, d3, 8, 0.0, 1.0, 4, buf, need, FAKE, None) == EINVAL
    assert st(FAKE, 1, d3, 8, 0.0, 1.0, 4, buf, need, None, None) == EINVAL
    assert st(FAKE, 5, d3, 8, 0.0, 1.0, 4, buf, need, FAKE, None) == EDTYPE
    assert st(FAKE, 1, dims(10, 0, 16), 8, 0.0, 1.0, 4, buf, need, FAKE, None) == EDIM
    assert st(FAKE, 1, d3, 8, 0.0, 1.0, 1, buf, need, FAKE, None) == EINVAL
    assert st(FAKE, 1, d3, 4097, 0.0, 1.0, 4, buf, need, FAKE, None) == ERANGE
    assert st(FAKE, 1, d3, 8, 1.0, 0.0, 4, buf, need, FAKE, None) == EINVAL
    assert st(FAKE, 1, d3, 8, 0.0, 1.0, 4, buf, need - 1, FAKE, None) == EWS
    assert st(FAKE, 1, d3, 8, 0.0, 1.0, 4, ctypes.c_void_p(0x100010), need, FAKE, None) == EWS


def test_binding_rejects_cpu_tensors():
    import torch

    with pytest.raises(TypeError):
        ecc.ecc_hard(torch.zeros(4, 4), 4, 0.0, 1.0)
    with pytest.raises(TypeError):
        ecc.ecc_soft_fwd(torch.zeros(4, 4), torch.zeros(3), 1.0, torch.ones(1), torch.zeros(2))


def test_debug_build_exports_every_declared_symbol():
    """The bounds-checked variant builds from the same sources, exports the same C ABI and says
    which build it is (no GPU needed for either)."""
    path = libbuild.build(debug=True)
    dbg = ctypes.CDLL(path)
    for n in declared_functions():
        assert hasattr(dbg, n), n
    dbg.ecc_debug_build.restype = ctypes.c_int
    assert dbg.ecc_debug_build() == 1
    rel = ecc.load_library()
    assert rel.ecc_debug_build() == 0
    assert rel.ecc_status_str(-8).startswith(b"ECC_EBOUNDS")
