"""The allocation-free soft-ECC forward entry point (ecc_soft_fwd_noalloc).

Some callers cannot allocate device memory -- a plugin inside a framework that owns all device
memory, or a latency-critical loop that cannot afford cudaMalloc's device-wide synchronisation.
For them the library keeps the soft-ECC forward workspace in its own fixed device array. These
tests call that entry point through the C ABI twice in a row, on different inputs, and compare
each result with the workspace-taking ecc_soft_fwd. Both run the same kernels on the same inputs,
so the results must be identical bit for bit: any stale data left in the shared array by the
previous call would show up as a difference. The file is collected last, and works both alone in
a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from euler_characteristic_curves_gb300 import ecc, synthetic

DEV = "cuda:0"
SCRATCH = 16 << 20  # ECC_NOALLOC_SCRATCH_BYTES
ERANGE = -6


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _same_bits(a, b):
    return torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.gpu
def test_noalloc_forward_matches_workspace_forward_twice():
    cases = [
        (synthetic.grf((128, 192), seed=41, batch=3), synthetic.uniform_thresholds(64), 50.0,
         synthetic.soft_direction(2, seed=42)),
        (synthetic.grf((256, 256), seed=43, batch=4), synthetic.uniform_thresholds(128, -0.1, 1.1),
         20.0, synthetic.soft_direction(2, seed=44)),
        # a smaller case after a larger one: the array still holds the previous call's entries
        (synthetic.grf((40, 70), seed=45, batch=2), synthetic.uniform_thresholds(16), 50.0,
         synthetic.soft_direction(2, seed=46)),
    ]
    for img, tau, lam, u in cases:
        x, t, a, uu = _dev(img), _dev(tau), torch.ones(1, device=DEV), _dev(u)
        ref, _ = ecc.ecc_soft_fwd(x, t, lam, a, uu)
        got = ecc.ecc_soft_fwd_noalloc(x, t, lam, a, uu)
        again = ecc.ecc_soft_fwd_noalloc(x, t, lam, a, uu)
        torch.cuda.synchronize()
        assert _same_bits(got, ref)
        assert _same_bits(again, ref)


@pytest.mark.gpu
def test_noalloc_largest_accepted_batch_and_first_rejected():
    """At K = 128 the forward workspace of 15 images of 256^2 fits the 16 MiB array and 16 do not:
    the largest accepted batch runs and matches the workspace forward bit for bit, the next one
    is rejected with ECC_ERANGE before anything runs."""
    lib = ecc.load_library()
    dims = (ctypes.c_int64 * 2)(256, 256)
    for batch in (15, 16):
        assert lib.ecc_soft_workspace_bytes(2, dims, batch, 128) > 0
    img = synthetic.grf((256, 256), seed=47, batch=15)
    x, t = _dev(img), _dev(synthetic.uniform_thresholds(128))
    a, uu = torch.ones(1, device=DEV), _dev(synthetic.soft_direction(2, seed=48))
    ref, _ = ecc.ecc_soft_fwd(x, t, 50.0, a, uu)
    got = ecc.ecc_soft_fwd_noalloc(x, t, 50.0, a, uu)
    torch.cuda.synchronize()
    assert _same_bits(got, ref)
    x16 = torch.cat([x, x[:1]])
    with pytest.raises(ecc.ECCError) as err:
        ecc.ecc_soft_fwd_noalloc(x16, t, 50.0, a, uu)
    assert err.value.status == ERANGE


@pytest.mark.gpu
def test_noalloc_rejects_sizes_beyond_its_array():
    lib = ecc.load_library()
    dims = (ctypes.c_int64 * 2)(1024, 1024)
    need = lib.ecc_soft_workspace_bytes(2, dims, 64, 128)
    assert need > SCRATCH
    fake = ctypes.c_void_p(0x100000)  # never dereferenced: the size check fails first
    rc = lib.ecc_soft_fwd_noalloc(fake, 2, dims, 64, fake, 128, 50.0, fake, fake, fake, None)
    assert rc == ERANGE
