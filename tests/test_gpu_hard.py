"""GPU parity for the hard ECC: the CUDA library (through the C ABI binding) against the CPU
oracle, bit-exact (int64), on seeded inputs.

Covers small shapes spanning several tiles with ragged tails, every special case the method has
(NaN, infinities, out-of-range values, ties, constant and checkerboard images, degenerate
threshold ranges, misaligned buffers, nbins from 1 to the maximum), 2-D and 3-D, uint8 and
float32, batches, and each benchmark workload at full size in the benchmark's launch
configuration (the library derives the launch from the sizes), 3-D launches whose blocks walk
several tasks in turn included. The oracle computes the largest volumes on every host core
(tests/_oracle_pool.py).
"""
import numpy as np
import pytest
import torch

import oracle
from euler_characteristic_curves_gb300 import ecc, synthetic
from tests import _oracle_pool

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def gpu_hard(img, nbins, vmin, vmax, ndim=None):
    if ndim is None:
        ndim = img.ndim  # an unbatched image or volume
    t = torch.from_numpy(np.ascontiguousarray(img)).to(DEV)
    return ecc.ecc_hard(t, nbins, vmin, vmax, ndim=ndim).cpu().numpy()


def check(img, nbins, vmin, vmax, ndim=None):
    got = gpu_hard(img, nbins, vmin, vmax, ndim)
    want = oracle.ecc_hard(img, nbins, vmin, vmax, ndim=ndim)
    np.testing.assert_array_equal(got, want)
    return got


def rand_field(shape, seed, kind="grf"):
    rng = np.random.default_rng(seed)
    if kind == "grf" and len(shape) >= 2 and min(shape) >= 2:
        return synthetic.grf(shape, seed)
    if kind == "ties":
        return rng.integers(0, 6, size=shape).astype(np.float32) / 5.0
    return rng.random(shape).astype(np.float32)


SIZES_H = [1, 2, 3, 5, 8, 17, 31, 32, 33, 67]
SIZES_W = [1, 2, 3, 4, 5, 7, 8, 31, 127, 128, 129, 131, 260, 515]


@pytest.mark.parametrize("h", SIZES_H)
def test_2d_size_sweep_f32(h):
    for i, w in enumerate(SIZES_W):
        for kind in ("grf", "ties"):
            f = rand_field((h, w), 100 * h + i, kind)
            check(f, 37, 0.0, 1.0)


@pytest.mark.parametrize("h", SIZES_H)
def test_2d_size_sweep_u8(h):
    rng = np.random.default_rng(h)
    for w in SIZES_W:
        q = rng.integers(0, 256, size=(h, w)).astype(np.uint8)
        check(q, 256, 0.0, 255.0)
        check(q // 40, 5, 0.0, 4.0)  # heavy ties
        check(q, 17, 30.0, 200.0)


def test_2d_batches_and_large_ragged():
    f = synthetic.grf((300, 517), 5, batch=3)
    check(f, 100, 0.0, 1.0, ndim=2)
    q = synthetic.quantise_u8(synthetic.grf((129, 1031), 6, batch=4))
    check(q, 256, 0.0, 255.0, ndim=2)
    f = synthetic.grf((1000, 1000), 7)
    check(f, 1024, 0.0, 1.0)


@pytest.mark.parametrize("nbins", [1023, 1024, 1025, 4096])
def test_nbins_variants_3d(nbins):
    """3-D at the boundary between the saturating flags (tables of up to 1024 bins) and the fp16
    compares (larger tables), f32 and uint8."""
    f = synthetic.grf((19, 37, 140), nbins)
    check(f, nbins, 0.0, 1.0)
    check(f, nbins, 0.3, 0.6)
    q = synthetic.quantise_u8(f)
    check(q, nbins, 0.0, 255.0)


@pytest.mark.parametrize("nbins", [1, 2, 3, 255, 256, 1000, 1024, 1025, 4096])
def test_nbins_variants(nbins):
    f = synthetic.grf((97, 203), nbins)
    check(f, nbins, 0.0, 1.0)
    check(f, nbins, 0.2, 0.7)
    q = synthetic.quantise_u8(f)
    check(q, nbins, 0.0, 255.0)


@pytest.mark.parametrize("shape,batch,nbins,kind", [((20, 37), 500, 100, "f32"),
                                                     ((20, 36), 500, 100, "f32"),
                                                     ((70, 260), 470, 1024, "f32"),
                                                     ((64, 130), 460, 256, "u8"),
                                                     ((9, 300), 470, 4096, "f32"),
                                                     ((3, 5), 600, 1, "f32"),
                                                     ((1, 1), 700, 7, "u8")])
def test_one_block_per_image_stores_the_curve_itself(shape, batch, nbins, kind):
    """A batch larger than the blocks that fit on the device at once gives each image a single
    block, which scans its own histogram and stores the curve (no zeroing, no atomics, no scan
    launch); every image must still match the oracle bit for bit."""
    f = synthetic.grf(shape, nbins + batch, batch=batch) if min(shape) > 1 else \
        np.random.default_rng(batch).random((batch,) + shape).astype(np.float32)
    if kind == "u8":
        check(synthetic.quantise_u8(f), nbins, 0.0, 255.0, ndim=2)
    else:
        check(f, nbins, 0.0, 1.0, ndim=2)


@pytest.mark.parametrize("shape,kind", [((3, 5), "f32"), ((4, 8), "f32"), ((2, 7), "u8"),
                                        ((2, 3, 4), "f32"), ((2, 2, 8), "u8")])
def test_hard_at_the_largest_batch(shape, kind):
    """65535 images or volumes (the grid's y extent), each its own block: every curve must match
    the oracle bit for bit. Rows of 8 values take the vector loads (2-D) and the TMA-staged
    kernel (3-D float32)."""
    rng = np.random.default_rng(sum(shape))
    f = rng.random((65535,) + shape).astype(np.float32)
    nd = len(shape)
    if kind == "u8":
        check(synthetic.quantise_u8(f), 256, 0.0, 255.0, ndim=nd)
    else:
        check(f, 17, 0.0, 1.0, ndim=nd)


def test_special_values():
    f = synthetic.grf((64, 160), 8)
    g = f.copy()
    g[3, 4] = np.nan
    g[10:13, 50:60] = np.inf
    g[20, :] = -np.inf
    g[30, 7] = 5.0
    g[40, 100] = -3.0
    g[63, 159] = np.nan
    g[0, 0] = np.nan
    check(g, 50, 0.0, 1.0)
    check(g, 50, -4.0, 6.0)
    check(np.full((33, 45), np.nan, np.float32), 10, 0.0, 1.0)
    check(np.full((33, 45), 0.5, np.float32), 11, 0.0, 1.0)
    check(np.full((33, 45), -0.0, np.float32), 3, -1.0, 0.0)
    z = np.zeros((16, 16), np.float32)
    z[::2, ::2] = -0.0
    check(z, 2, -1.0, 0.0)
    cb = (np.indices((41, 66)).sum(0) % 2).astype(np.float32)
    check(cb, 2, 0.0, 1.0)
    check(cb.astype(np.uint8), 2, 0.0, 1.0)
    check(1.0 - cb, 3, 0.0, 1.0)


def test_2d_vector_rows_special_cases():
    """2-D float32 images with rows of a multiple of 4 values (each lane reads its four values
    with one load) on the cases that decide the flags and keys: ties broken by position
    (checkerboards, quantised values, constants), values on and one ulp around every threshold
    (the exact fix-up of ambiguous estimates), NaN and infinities, strips and row ranges with
    ragged ends, and the largest table of the saturating flags."""
    cb = (np.indices((41, 68)).sum(0) % 2).astype(np.float32)
    check(cb, 2, 0.0, 1.0)
    check(1.0 - cb, 3, 0.0, 1.0)
    check(np.full((33, 44), np.nan, np.float32), 10, 0.0, 1.0)
    check(np.full((33, 44), 0.5, np.float32), 11, 0.0, 1.0)
    check(rand_field((65, 132), 3, "ties"), 6, 0.0, 1.0)
    H = 64
    t = oracle.thresholds(H, 0.0, 1.0)
    vals = []
    for x in t:
        x32 = np.float32(x)
        vals += [np.nextafter(x32, np.float32(-1)), x32, np.nextafter(x32, np.float32(2))]
    rng = np.random.default_rng(19)
    check(rng.choice(np.asarray(vals, np.float32), size=(50, 76)).astype(np.float32), H, 0.0, 1.0)
    check(rng.choice(np.arange(1024, dtype=np.float32), size=(90, 260)), 1024, 0.0, 1023.0)
    g = synthetic.grf((97, 388), 20)
    g[0, :] = np.nan
    g[:, 127:129] = np.inf
    g[31:33, :] = -np.inf
    g[96, 387] = np.nan
    check(g, 1024, 0.0, 1.0)
    check(g, 1, 0.0, 1.0)
    check(synthetic.grf((300, 516), 22, batch=3), 100, 0.0, 1.0, ndim=2)


def test_threshold_edges_exact():
    # values that sit exactly on, or one ulp around, every threshold
    H = 64
    t = oracle.thresholds(H, 0.0, 1.0)
    vals = []
    for x in t:
        x32 = np.float32(x)
        vals += [np.nextafter(x32, np.float32(-1)), x32, np.nextafter(x32, np.float32(2))]
    vals = np.asarray(vals, np.float32)
    rng = np.random.default_rng(9)
    img = rng.choice(vals, size=(50, 77)).astype(np.float32)
    check(img, H, 0.0, 1.0)
    img = rng.choice(np.arange(256, dtype=np.float32), size=(50, 77))
    check(img, 256, 0.0, 255.0)  # integer thresholds: exact ties with data


def test_degenerate_and_badly_conditioned_ranges():
    f = synthetic.grf((40, 90), 10)
    check(f, 5, 0.5, 0.5)  # all thresholds equal
    check(f, 1, 0.25, 0.25)
    big = (f.astype(np.float64) * 1e-3 + 1000.0).astype(np.float32)
    check(big, 1024, 1000.0, 1000.001)  # offset >> range: search mode
    check(big, 700, 1000.0002, 1000.0009)
    check(-f, 200, -1.0, 0.0)
    check(f * 3e38, 100, 0.0, 3e38)
    check(f * 1e-38, 100, 0.0, 1e-38)  # subnormal thresholds


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_misaligned_buffers(offset):
    f = synthetic.grf((37, 128), 11 + offset)
    base = torch.zeros(f.size + 8, dtype=torch.float32, device=DEV)
    view = base[offset: offset + f.size].view(37, 128)
    view.copy_(torch.from_numpy(f).to(DEV))
    got = ecc.ecc_hard(view, 64, 0.0, 1.0).cpu().numpy()
    np.testing.assert_array_equal(got, oracle.ecc_hard(f, 64, 0.0, 1.0))
    q = synthetic.quantise_u8(f)
    b8 = torch.zeros(q.size + 8, dtype=torch.uint8, device=DEV)
    v8 = b8[offset: offset + q.size].view(37, 128)
    v8.copy_(torch.from_numpy(q).to(DEV))
    got = ecc.ecc_hard(v8, 256, 0.0, 255.0).cpu().numpy()
    np.testing.assert_array_equal(got, oracle.ecc_hard(q, 256, 0.0, 255.0))


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_misaligned_volumes(offset):
    """3-D float32 volumes whose rows hold a multiple of 4 values but whose base is not 16-byte
    aligned: the TMA-staged kernel's tensor map needs the aligned base, so these take the
    register-prefetch kernel, and must match the oracle like the aligned ones (uint8 too)."""
    v = synthetic.grf((6, 40, 132), 70 + offset)
    base = torch.zeros(v.size + 8, dtype=torch.float32, device=DEV)
    view = base[offset: offset + v.size].view(v.shape)
    view.copy_(torch.from_numpy(v).to(DEV))
    got = ecc.ecc_hard(view, 64, 0.0, 1.0, ndim=3).cpu().numpy()
    np.testing.assert_array_equal(got, oracle.ecc_hard(v, 64, 0.0, 1.0))
    q = synthetic.quantise_u8(v)
    b8 = torch.zeros(q.size + 8, dtype=torch.uint8, device=DEV)
    v8 = b8[offset: offset + q.size].view(q.shape)
    v8.copy_(torch.from_numpy(q).to(DEV))
    got = ecc.ecc_hard(v8, 256, 0.0, 255.0, ndim=3).cpu().numpy()
    np.testing.assert_array_equal(got, oracle.ecc_hard(q, 256, 0.0, 255.0))


@pytest.mark.parametrize("shape", [(1, 1, 1), (2, 2, 2), (3, 1, 7), (1, 9, 9), (5, 6, 7),
                                   (9, 17, 33), (4, 8, 128), (3, 9, 129), (17, 20, 131),
                                   (2, 67, 260), (40, 12, 5)])
def test_3d_shapes(shape):
    for kind in ("grf", "ties", "uniform"):
        v = rand_field(shape, sum(shape), kind)
        check(v, 29, 0.0, 1.0)
        check(synthetic.quantise_u8(v), 256, 0.0, 255.0)


def test_3d_batches_special_values():
    v = synthetic.grf((12, 20, 44), 12, batch=3)
    v[0, 3, 4, 5] = np.nan
    v[1, :, 7, :] = np.inf
    v[2, 5] = -np.inf
    check(v, 64, 0.0, 1.0, ndim=3)
    q = synthetic.quantise_u8(synthetic.grf((7, 33, 64), 13, batch=2))
    check(q, 256, 0.0, 255.0, ndim=3)
    check(q, 9, 100.0, 140.0, ndim=3)


def test_calls_without_a_stream_use_the_current_stream():
    assert ecc._stream_handle(None) == torch.cuda.current_stream().cuda_stream
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        assert ecc._stream_handle(None) == s.cuda_stream != torch.cuda.default_stream().cuda_stream
        f = synthetic.grf((70, 90), 15)
        got = ecc.ecc_hard(torch.from_numpy(f).to(DEV), 33, 0.0, 1.0)
    s.synchronize()
    np.testing.assert_array_equal(got.cpu().numpy(), oracle.ecc_hard(f, 33, 0.0, 1.0))


def test_deterministic_and_stream_independent():
    f = synthetic.grf((333, 444), 14)
    t = torch.from_numpy(f).to(DEV)
    a = ecc.ecc_hard(t, 512, 0.0, 1.0)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = ecc.ecc_hard(t, 512, 0.0, 1.0, stream=s)
    s.synchronize()
    assert torch.equal(a, b)


# ------------------------------------------------------------------------ full-size workloads

def test_workload_128sq_u8():
    img = synthetic.blurred_noise_u8((128, 128), seed=1, sigma=3.0)
    check(img, 256, 0.0, 255.0)


def test_workload_16x1024sq_f32():
    img = synthetic.grf((1024, 1024), seed=2, batch=16)
    check(img, 256, 0.0, 1.0, ndim=2)


def test_workload_8192sq_f32():
    img = synthetic.grf((8192, 8192), seed=3)
    check(img, 1024, 0.0, 1.0)


def test_workload_512cube_u8():
    v = synthetic.grf((512, 512, 512), seed=5, device=DEV)
    q = synthetic.quantise_u8(v)
    got = ecc.ecc_hard(q.unsqueeze(0), 256, 0.0, 255.0).cpu().numpy()[0]
    want = oracle.ecc_hard(q.cpu().numpy(), 256, 0.0, 255.0)
    np.testing.assert_array_equal(got, want)


def test_workload_1024cube_f32():
    """The 1024^3 volume in the benchmark's launch -- 57 groups of 8 side-by-side blocks, each
    group a contiguous segment of the 32 rows of tiles x 1024 planes in up to two pieces (tasks),
    so blocks carry their key buffers and histogram from one piece to the next -- against the
    oracle, bit for bit. The oracle curve comes from slabs that share one plane, one oracle
    process per host core."""
    v = synthetic.grf((1024, 1024, 1024), seed=4, device=DEV)
    plan = ecc.hard_launch_info(tuple(v.shape), 1, 256)
    assert plan["rounds"] > 1 and plan["tasks_per_image"] > plan["blocks_per_image"]
    got = ecc.ecc_hard(v.unsqueeze(0), 256, 0.0, 1.0)[0].cpu().numpy()
    want = _oracle_pool.hard_volume(v.cpu().numpy(), 256, 0.0, 1.0)
    np.testing.assert_array_equal(got, want)
    assert got[-1] == 1


@pytest.mark.parametrize("shape,kind,nbins", [((16, 2048, 2048), "f32", 256),
                                              ((64, 1024, 1024), "f32", 1000),
                                              ((32, 1024, 1024), "u8", 256)])
def test_3d_blocks_walking_several_tasks(shape, kind, nbins):
    """Volumes where each block walks several tasks, reusing its key ring, carried rows and
    histogram from one to the next: float32 with 256 bins (the TMA-staged kernel: 28 groups of 16
    side-by-side blocks, each a segment of the 64 rows of tiles x 16 planes in up to four
    pieces), float32 with 1000 bins and uint8
    (the register-prefetch kernel, 456 blocks taking (tile, chunk) tasks in rounds). The planner
    says how many tasks a block walks; the curve must match the oracle bit for bit."""
    v = synthetic.grf(shape, seed=30 + shape[0], device=DEV)
    vmax = 1.0
    if kind == "u8":
        v, vmax = synthetic.quantise_u8(v), 255.0
    plan = ecc.hard_launch_info(tuple(v.shape), 1, nbins, dtype=v.dtype)
    assert plan["rounds"] > 1, plan
    got = ecc.ecc_hard(v.unsqueeze(0), nbins, 0.0, vmax)[0].cpu().numpy()
    want = _oracle_pool.hard_volume(v.cpu().numpy(), nbins, 0.0, vmax)
    np.testing.assert_array_equal(got, want)


def test_3d_rounds_on_a_small_device_plan():
    """Blocks walking several tasks on small volumes: a batch of 100 volumes shares the resident
    blocks, so each image gets a few blocks and more tiles than blocks (checked with the
    planner), ragged tiles included; float32 (TMA-staged kernel: segments in several pieces)
    and uint8 (register-prefetch kernel: tasks in rounds)."""
    v = synthetic.grf((8, 70, 300), seed=33, batch=100)
    assert ecc.hard_launch_info(v.shape[1:], 100, 77)["rounds"] > 1
    check(v, 77, 0.0, 1.0, ndim=3)
    q = synthetic.quantise_u8(v)
    assert ecc.hard_launch_info(v.shape[1:], 100, 256, dtype=torch.uint8)["rounds"] > 1
    check(q, 256, 0.0, 255.0, ndim=3)


def test_library_calls_replay_from_a_cuda_graph():
    """Calls are asynchronous on the current stream and allocate nothing on the device, so they
    capture into a CUDA graph; a replay after the inputs change in place must give what eager
    calls give on the new inputs (hard 2-D with one block per image, hard 3-D, soft fwd + bwd)."""
    img2 = torch.from_numpy(synthetic.grf((96, 200), 21, batch=3)).to(DEV)
    vol = torch.from_numpy(synthetic.grf((20, 40, 150), 22)).to(DEV)
    simg = torch.from_numpy(synthetic.grf((64, 64), 23, batch=2)).to(DEV)
    tau = torch.from_numpy(synthetic.uniform_thresholds(32)).to(DEV)
    alpha = torch.ones(1, device=DEV)
    u = torch.from_numpy(synthetic.soft_direction(2, 24)).to(DEV)
    g = torch.from_numpy(synthetic.upstream_grad((2, 32), 25)).to(DEV)
    o2 = torch.empty((3, 77), dtype=torch.int64, device=DEV)
    o3 = torch.empty((1, 64), dtype=torch.int64, device=DEV)
    ws = torch.empty(ecc.soft_workspace_bytes((64, 64), 2, 32), dtype=torch.uint8, device=DEV)
    s_out = torch.empty((2, 32), dtype=torch.float32, device=DEV)

    def calls():
        ecc.ecc_hard(img2, 77, 0.0, 1.0, ndim=2, out=o2)
        ecc.ecc_hard(vol.unsqueeze(0), 64, 0.0, 1.0, out=o3)
        ecc.ecc_soft_fwd(simg, tau, 50.0, alpha, u, ws=ws, out=s_out)
        return ecc.ecc_soft_bwd(simg, tau, 50.0, alpha, u, g, ws)

    calls()  # warm-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        grads = calls()
    for seed in (26, 27):
        img2.copy_(torch.from_numpy(synthetic.grf((96, 200), seed, batch=3)))
        vol.copy_(torch.from_numpy(synthetic.grf((20, 40, 150), seed)))
        simg.copy_(torch.from_numpy(synthetic.grf((64, 64), seed, batch=2)))
        graph.replay()
        torch.cuda.synchronize()
        got = [o2.clone(), o3.clone(), s_out.clone()] + [grads[k].clone() for k in sorted(grads)]
        want_g = calls()
        torch.cuda.synchronize()
        want = [o2, o3, s_out] + [want_g[k] for k in sorted(want_g)]
        for a, b in zip(got, want):
            assert torch.equal(a, b)
        np.testing.assert_array_equal(got[0].cpu().numpy(),
                                      oracle.ecc_hard(img2.cpu().numpy(), 77, 0.0, 1.0, ndim=2))
