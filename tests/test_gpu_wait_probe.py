"""The failure path of the kernels' bounded waits, made to run out on purpose without a fault.

The TMA-staged kernels wait for each staged copy on an mbarrier with a time limit; past it a
kernel records a timeout in the device error word and returns instead of hanging. The probe
(ecc_wait_probe) runs that same bounded wait, cut to a short limit, on an mbarrier that nothing
arrives at: the test checks that the wait really ran its limit, that the host reads
ECC_ETIMEOUT from ecc_device_status, that reading clears it, and that the context still
computes correct curves afterwards.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from euler_characteristic_curves_gb300 import ecc, synthetic

pytestmark = pytest.mark.gpu
ECC_OK, ECC_ETIMEOUT = 0, -7


def test_a_wait_that_runs_out_reports_timeout_and_the_context_stays_usable():
    torch.cuda.synchronize()
    assert ecc.device_status() == ECC_OK  # clears anything earlier
    limit_s = 0.05
    t0 = time.perf_counter()
    ecc.wait_probe(int(limit_s * 1e9))
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert limit_s <= waited < 2.0, waited
    assert ecc.device_error_bits(clear=False) & 1
    assert ecc.device_status() == ECC_ETIMEOUT  # and cleared
    assert ecc.device_status() == ECC_OK
    # the context is still usable: a 3-D call (the TMA-staged kernel) and a 2-D call match
    vol = synthetic.grf((9, 40, 132), 44)
    got = ecc.ecc_hard(torch.from_numpy(vol).cuda(), 64, 0.0, 1.0, ndim=3).cpu().numpy()
    np.testing.assert_array_equal(got, oracle.ecc_hard(vol, 64, 0.0, 1.0))
    img = synthetic.grf((70, 90), 45)
    got = ecc.ecc_hard(torch.from_numpy(img).cuda(), 33, 0.0, 1.0).cpu().numpy()
    np.testing.assert_array_equal(got, oracle.ecc_hard(img, 33, 0.0, 1.0))
    assert ecc.device_status() == ECC_OK
