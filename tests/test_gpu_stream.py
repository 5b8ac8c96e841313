"""GPU parity for the streamed hard ECC of volumes read in slabs of planes (bit-exact against the
oracle, and against the device-resident path where the oracle would be slow)."""
import numpy as np
import pytest
import torch

import oracle
from euler_characteristic_curves_gb300 import ecc, synthetic

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def volume(shape, seed, kind):
    v = synthetic.grf(shape, seed)
    if kind == "u8":
        return synthetic.quantise_u8(v)
    return v


def host(a, pinned):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.pin_memory() if pinned else t


@pytest.mark.parametrize("kind,nbins,vmax", [("f32", 64, 1.0), ("u8", 256, 255.0)])
@pytest.mark.parametrize("slab", [2, 3, 7, 40, 64])
def test_stream_matches_oracle(kind, nbins, vmax, slab):
    v = volume((40, 33, 70), seed=slab, kind=kind)
    got = ecc.ecc_hard_stream(host(v, pinned=True), nbins, 0.0, vmax, slab_planes=slab)
    want = oracle.ecc_hard(v, nbins, 0.0, vmax)
    np.testing.assert_array_equal(got.cpu().numpy(), want)


@pytest.mark.parametrize("shape", [(1, 9, 12), (2, 5, 6), (3, 1, 1), (5, 130, 3), (17, 8, 128)])
def test_stream_edge_shapes(shape):
    v = volume(shape, seed=sum(shape), kind="f32") if min(shape) > 1 else \
        np.random.default_rng(4).random(shape).astype(np.float32)
    for slab in (2, 4):
        got = ecc.ecc_hard_stream(host(v, pinned=False), 32, 0.0, 1.0, slab_planes=slab)
        np.testing.assert_array_equal(got.cpu().numpy(), oracle.ecc_hard(v, 32, 0.0, 1.0))


def test_stream_nan_inf_and_every_source_memory():
    v = volume((12, 20, 36), seed=5, kind="f32")
    v[3, 4, 5] = np.nan
    v[6, :, 7] = np.inf
    v[9] = -np.inf
    want = oracle.ecc_hard(v, 40, 0.0, 1.0)
    for src in (host(v, True), host(v, False), torch.from_numpy(v).to(DEV)):
        got = ecc.ecc_hard_stream(src, 40, 0.0, 1.0, slab_planes=5)
        np.testing.assert_array_equal(got.cpu().numpy(), want)


def test_stream_256x512sq_matches_resident_and_reuses_buffers():
    """A 256 MB volume in 32-plane slabs, twice with the same buffers, against ecc_hard on the
    resident volume (itself checked against the oracle in test_gpu_hard.py)."""
    v = synthetic.grf((256, 512, 512), 4, device=DEV)
    resident = ecc.ecc_hard(v.unsqueeze(0), 256, 0.0, 1.0, ndim=3)[0]
    h = v.cpu().pin_memory()
    buf = torch.empty(ecc.hard_stream_buffer_bytes(tuple(v.shape), v.dtype, 32),
                      dtype=torch.uint8, device=DEV)
    for _ in range(2):
        got = ecc.ecc_hard_stream(h, 256, 0.0, 1.0, slab_planes=32, buf=buf)
        assert torch.equal(got, resident)
    # a sampled slab of the same volume against the oracle (planes 100..131)
    sub = v[100:132].contiguous()
    got = ecc.ecc_hard_stream(sub.cpu().pin_memory(), 256, 0.0, 1.0, slab_planes=9)
    np.testing.assert_array_equal(got.cpu().numpy(),
                                  oracle.ecc_hard(sub.cpu().numpy(), 256, 0.0, 1.0))
