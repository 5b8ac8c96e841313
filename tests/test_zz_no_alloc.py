"""The allocation-free soft-ECC forward entry point (ecc_soft_fwd_noalloc).

Some callers cannot allocate device memory -- a plugin inside a framework that owns all device
memory, or a latency-critical loop that cannot afford cudaMalloc's device-wide synchronisation.
For them the library keeps the soft-ECC workspace in its own fixed device array. This test calls
that entry point through the C ABI twice in a row, on different inputs, and checks each result
against the workspace-taking ecc_soft_fwd with the soft path's tolerance (1e-6 absolute plus
1e-4 relative). It lives in its own file, collected last, and works both alone in a fresh process
and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from euler_characteristic_curves_gb300 import ecc, synthetic

DEV = "cuda:0"


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


@pytest.mark.gpu
def test_noalloc_forward_matches_workspace_forward_twice():
    cases = [
        (synthetic.grf((128, 192), seed=41, batch=3), synthetic.uniform_thresholds(64), 50.0,
         synthetic.soft_direction(2, seed=42)),
        (synthetic.grf((256, 256), seed=43, batch=4), synthetic.uniform_thresholds(128, -0.1, 1.1),
         20.0, synthetic.soft_direction(2, seed=44)),
    ]
    for img, tau, lam, u in cases:
        x, t, a, uu = _dev(img), _dev(tau), torch.ones(1, device=DEV), _dev(u)
        ref, _ = ecc.ecc_soft_fwd(x, t, lam, a, uu)
        got = ecc.ecc_soft_fwd_noalloc(x, t, lam, a, uu)
        torch.cuda.synchronize()
        ref, got = ref.double().cpu().numpy(), got.double().cpu().numpy()
        assert np.all(np.abs(got - ref) <= 1e-6 + 1e-4 * np.abs(ref))


@pytest.mark.gpu
def test_noalloc_rejects_sizes_beyond_its_array():
    lib = ecc.load_library()
    dims = (ctypes.c_int64 * 2)(1024, 1024)
    need = lib.ecc_soft_workspace_bytes(2, dims, 64, 128)
    assert need > (16 << 20)
    fake = ctypes.c_void_p(0x100000)  # never dereferenced: the size check fails first
    rc = lib.ecc_soft_fwd_noalloc(fake, 2, dims, 64, fake, 128, 50.0, fake, fake, fake, None)
    assert rc == -6  # ECC_ERANGE
