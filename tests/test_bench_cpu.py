"""bench.py's host-side contract, on the CPU: the reference arm's JSON line (the oracle timed on
the host), the warm-up rule, and the per-part kernel launch count the line reports."""
import contextlib
import io
import json

import pytest

import bench


def test_reference_arm_prints_one_complete_json_line():
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--workload", "2d128u8", "--steps", "1",
                         "--warmup", "3"])
    assert rc == 0
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True and d["vs_baseline"] is None
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["unit"] == d["unit"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] and d["config"]["parts"] == ["hard_2d_1x128x128_u8blur_H256"]


def test_warmup_below_three_is_refused():
    with pytest.raises(SystemExit):
        with contextlib.redirect_stderr(io.StringIO()):
            bench.main(["--impl", "reference", "--workload", "2d128u8", "--warmup", "2"])


def test_hard_launch_count_per_part():
    """A 3-D call launches the pass and the scan; a 2-D call the pass alone (its blocks add the
    running sums of their histograms, or an image's only block stores its curve); a streamed
    volume launches a 3-D pass per slab, a plane pass from the second slab on and one scan."""
    w = bench.WORKLOADS
    assert [bench.hard_launches(p, 152) for p in w["headline"] if p[0] == "hard"] == [1, 2]
    assert bench.hard_launches(w["2d128u8"][0], 152) == 1
    assert bench.hard_launches(w["2d1024x16"][0], 152) == 1
    assert bench.hard_launches(w["3d512u8"][0], 152) == 2
    stream = w["3d1024stream"][0]
    slab = bench.part_slab(stream)
    # slabs of `slab` planes sharing one plane: ceil((D - 1) / (slab - 1)) of them
    n = -(-(stream[1][0] - 1) // (slab - 1))
    assert bench.hard_launches(stream, 152) == 2 * n
    # a batch larger than the resident blocks gives every image its own single block
    big_batch = ("hard", (1024, 1024), 1000, "f32", 256, 0.0, 1.0, 2)
    assert bench.hard_launches(big_batch, 152) == 1


def test_sharded_workload_reference_line_and_plan():
    """The sharded-volume workload: its reference line reports strong scaling, and its
    per-rank algorithmic bytes follow the slab plan (every plane once, the shared ones twice)."""
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        assert bench.main(["--impl", "reference", "--workload", "3d1024shard", "--steps", "1",
                           "--warmup", "3"]) == 0
    d = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert d["scaling"] == "strong" and d["value"] > 0
    p = bench.WORKLOADS["3d1024shard"][0]
    assert bench.hard_kernel_name(p) == "ecc_hard3d_tma_kernel"
    for world in (1, 2, 4, 8):
        planes = [bench.time_inputs_planes(p, r, world) for r in range(world)]
        assert sum(planes) == 1024 + world - 1
        assert bench.part_alg_bytes(p, planes[0]) == planes[0] * 1024 * 1024 * 4 + 8 * 256
