"""Small parity cases under the bounds-checked debug build (test infrastructure).

Run in a process of its own with ECC_DEBUG=1, so that the binding loads the debug variant of the
library: every case is compared with the oracle, then the device error word must be clean (no
bounds check failed, no wait gave up). Prints one line "debug-run ok <bits>" on success.
"""
import sys

import numpy as np
import torch

import oracle
from euler_characteristic_curves_gb300 import ecc, synthetic

DEV = "cuda:0"


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def main():
    lib = ecc.load_library()
    assert lib.ecc_debug_build() == 1, "ECC_DEBUG=1 must load the debug build"
    ecc.device_status(clear=True)
    # hard 2-D: ragged strips, several blocks (prefix flush), one block (direct), u8, search mode
    for shape, nb, batch in [((67, 133), 64, None), ((300, 517), 100, 3), ((31, 260), 1024, 2)]:
        f = synthetic.grf(shape, sum(shape), batch=batch)
        got = ecc.ecc_hard(dev(f), nb, 0.0, 1.0, ndim=2).cpu().numpy()
        np.testing.assert_array_equal(got, oracle.ecc_hard(f, nb, 0.0, 1.0, ndim=2))
    q = synthetic.quantise_u8(synthetic.grf((129, 1031), 6, batch=2))
    np.testing.assert_array_equal(ecc.ecc_hard(dev(q), 256, 0.0, 255.0, ndim=2).cpu().numpy(),
                                  oracle.ecc_hard(q, 256, 0.0, 255.0, ndim=2))
    big = (synthetic.grf((40, 90), 10).astype(np.float64) * 1e-3 + 1000.0).astype(np.float32)
    np.testing.assert_array_equal(ecc.ecc_hard(dev(big), 700, 1000.0002, 1000.0009).cpu().numpy(),
                                  oracle.ecc_hard(big, 700, 1000.0002, 1000.0009))
    # hard 3-D: TMA-staged (f32, W % 4 == 0), register kernel (odd W, u8, > 256 bins), batches
    for shape, nb in [((10, 40, 140), 100), ((9, 17, 33), 29), ((19, 37, 140), 1025)]:
        v = synthetic.grf(shape, sum(shape) + nb)
        np.testing.assert_array_equal(ecc.ecc_hard(dev(v), nb, 0.0, 1.0, ndim=3).cpu().numpy(),
                                      oracle.ecc_hard(v, nb, 0.0, 1.0))
        u8 = synthetic.quantise_u8(v)
        np.testing.assert_array_equal(
            ecc.ecc_hard(dev(u8), 256, 0.0, 255.0, ndim=3).cpu().numpy(),
            oracle.ecc_hard(u8, 256, 0.0, 255.0))
    vb = synthetic.grf((8, 70, 300), 33, batch=100)
    np.testing.assert_array_equal(ecc.ecc_hard(dev(vb), 77, 0.0, 1.0, ndim=3).cpu().numpy(),
                                  oracle.ecc_hard(vb, 77, 0.0, 1.0, ndim=3))
    # streamed and partial (sharded) paths
    w = synthetic.grf((10, 40, 140), 6)
    np.testing.assert_array_equal(
        ecc.ecc_hard_stream(torch.from_numpy(w), 100, 0.0, 1.0, slab_planes=4).cpu().numpy(),
        oracle.ecc_hard(w, 100, 0.0, 1.0))
    # soft forward and backward, 2-D and 3-D, and the transform
    for shape, K in [((40, 70), 16), ((12, 20, 45), 129)]:
        img = synthetic.grf(shape, K, batch=2)
        tau = synthetic.uniform_thresholds(K, -0.2, 1.2)
        u = synthetic.soft_direction(len(shape), K)
        g = synthetic.upstream_grad((2, K), K + 1)
        a = np.asarray([1.0], np.float32)
        s, ws = ecc.ecc_soft_fwd(dev(img), dev(tau), 50.0, dev(a), dev(u))
        res = ecc.ecc_soft_bwd(dev(img), dev(tau), 50.0, dev(a), dev(u), dev(g), ws,
                               want_img=True)
        ref = oracle.ecc_soft_fwd(img, tau, 50.0, 1.0, u, ndim=len(shape))
        assert np.all(np.abs(s.cpu().numpy() - ref) <= 1e-6 + 1e-4 * np.abs(ref))
        rb = oracle.ecc_soft_bwd(img, tau, 50.0, 1.0, u, g, ndim=len(shape), want_img=False)
        gt = res["grad_tau"].cpu().numpy()
        assert np.all(np.abs(gt - rb["grad_tau"]) <= 1e-6 + 1e-4 * np.abs(rb["grad_tau"]))
    U = np.stack([synthetic.soft_direction(2, 60 + j) for j in range(3)])
    img = synthetic.grf((33, 65), 61, batch=2)
    tau = synthetic.uniform_thresholds(24)
    S, ws = ecc.ecc_soft_ect_fwd(dev(img), dev(tau), 50.0, torch.ones(1, device=DEV), dev(U))
    ref = oracle.ecc_soft_ect_fwd(img, tau, 50.0, 1.0, U, ndim=2)
    assert np.all(np.abs(S.cpu().numpy() - ref) <= 1e-6 + 1e-4 * np.abs(ref))
    torch.cuda.synchronize()
    bits = ecc.device_error_bits(clear=True)
    assert bits == 0, f"device error bits {bits:#x} after the debug-build cases"
    print(f"debug-run ok {bits}")
    return 0


if __name__ == "__main__":
    sys.exit(main())
