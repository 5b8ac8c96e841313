"""Benchmark of the ECC hot path on GB300 (prints one JSON line on rank 0).

A step is one pass of the whole hot path over one batch of synthetic input, inputs resident in
HBM: the hard ECC of the 2-D 8192^2 float32 image (nbins 1024) and of the 3-D 1024^3 float32
volume (nbins 256) -- the two grids the headline metric is quoted on -- plus the soft ECC
forward and backward on 64 images of 256^2 (K = 128, lambda = 50). ``value`` is hard-ECC
Gvoxels per second of the whole step; the per-part device times, the roofline fraction of the
dominant kernel and the soft fwd+bwd milliseconds are reported beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload headline|2d8192|3d1024|2d1024x16|2d128u8|3d512u8|soft|soft3d]

Under torchrun every rank runs the same workload on its own GPU (independent problems, no
collective on the data path; weak scaling); the timed region is bracketed by barriers and the
slowest rank's time is reported. ``--impl reference`` times the CPU oracle (the plain C
definition) on a bounded sample of the same workload on this host's cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("Gvoxels/s hard ECC (2D 8192^2, 3D 1024^3) as % HBM roofline; "
          "soft-ECC fwd+bwd ms")

# ------------------------------------------------------------------------------------ workloads

WORKLOADS = {
    # name: list of parts; a part is ("hard", shape, batch, dtype, nbins, vmin, vmax, seed) or
    # ("soft", shape, batch, K, lam, seed_img, seed_u, seed_g)
    "2d128u8": [("hard", (128, 128), 1, "u8blur", 256, 0.0, 255.0, 1)],
    "2d1024x16": [("hard", (1024, 1024), 16, "f32", 256, 0.0, 1.0, 2)],
    "2d8192": [("hard", (8192, 8192), 1, "f32", 1024, 0.0, 1.0, 3)],
    "3d1024": [("hard", (1024, 1024, 1024), 1, "f32", 256, 0.0, 1.0, 4)],
    "3d512u8": [("hard", (512, 512, 512), 1, "u8grf", 256, 0.0, 255.0, 5)],
    "soft": [("soft", (256, 256), 64, 128, 50.0, 6, 7, 8)],
    # smaller cases of the same kernels (inputs still larger than L2) for ncu captures
    "3d256": [("hard", (256, 1024, 1024), 1, "f32", 256, 0.0, 1.0, 4)],
    "2d4096": [("hard", (4096, 4096), 1, "f32", 1024, 0.0, 1.0, 3)],
    "soft16": [("soft", (256, 256), 16, 128, 50.0, 6, 7, 8)],
    # the soft path on 3-D volumes (3 x 3 x 3 neighbourhoods): 4 GRF volumes of 128^3
    "soft3d": [("soft", (128, 128, 128), 4, 128, 50.0, 9, 10, 11)],
    # the soft Euler characteristic transform: 16 GRF images of 256^2 along 32 directions
    # (a soft part with a ninth field, the number of directions)
    "ect": [("soft", (256, 256), 16, 128, 50.0, 12, 13, 14, 32)],
    # the 1024^3 volume streamed from page-locked host memory in 64-plane slabs (a hard part
    # with a ninth field, the slab length): the out-of-core path, bound by the host link
    "3d1024stream": [("hard", (1024, 1024, 1024), 1, "f32", 256, 0.0, 1.0, 4, 64)],
    # the 1024^3 volume sharded over the ranks in slabs that share one plane: each rank adds its
    # slab's partial histogram, one all-reduce of 256 int64, one running sum (strong scaling)
    "3d1024shard": [("shard", (1024, 1024, 1024), 1, "f32", 256, 0.0, 1.0, 4)],
}
WORKLOADS["headline"] = WORKLOADS["2d8192"] + WORKLOADS["3d1024"] + WORKLOADS["soft"]

DESCRIPTION = {
    "headline": "hard ECC 2D 8192^2 f32 nbins 1024 + 3D 1024^3 f32 nbins 256; "
                "soft ECC fwd+bwd 64x256^2 f32 K 128 lambda 50",
}


def part_slab(p):
    """Slab length of a streamed hard part (0: the volume is resident on the device)."""
    return p[8] if p[0] == "hard" and len(p) > 8 else 0


def part_dirs(p):
    """Directions of a soft part (1 for the soft ECC, more for the transform)."""
    return p[8] if p[0] == "soft" and len(p) > 8 else 1


def part_name(p):
    if p[0] == "shard":
        return f"hard_3d_sharded_{'x'.join(str(s) for s in p[1])}_{p[3]}_H{p[4]}"
    if p[0] == "hard":
        dims = "x".join(str(s) for s in p[1])
        return f"hard_{len(p[1])}d_{p[2]}x{dims}_{p[3]}_H{p[4]}"
    name = f"soft_fwd_bwd_{p[2]}x{'x'.join(str(x) for x in p[1])}_K{p[3]}"
    return name if part_dirs(p) == 1 else name.replace("soft_", "soft_ect_") + f"_D{part_dirs(p)}"


def hard_kernel_name(p):
    """The library's kernel for a hard part: the TMA-staged 3-D kernel for float32 volumes with
    rows of a multiple of 4 values and at most 256 bins, else the register-prefetch 3-D kernel or
    the 2-D kernel."""
    if len(p[1]) == 2:
        return "ecc_hard2d_kernel"
    if p[3] == "f32" and p[4] <= 256 and p[1][-1] % 4 == 0:
        return "ecc_hard3d_tma_kernel"
    return "ecc_hard3d_kernel"


def time_inputs_planes(p, rank, world):
    """Planes this rank processes of a sharded part (None for other parts)."""
    if p[0] != "shard":
        return None
    from euler_characteristic_curves_gb300 import shard

    a, b = shard.slab_plan(p[1][0], world)[rank]
    return b - a + 1


def part_alg_bytes(p, planes=None):
    """Algorithmic bytes of a hard part per call on this rank: every voxel read once, one int64
    per (image, bin) written. A sharded part counts this rank's slab."""
    elem = 1 if p[3].startswith("u8") else 4
    vox = part_voxels(p)
    if planes is not None:
        vox = vox // p[1][0] * planes
    return vox * elem + 8 * p[2] * p[4]


def part_voxels(p):
    n = p[2]
    for s in p[1]:
        n *= s
    return n


# ------------------------------------------------------------------------------------ helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# Sources that make up the hard kernels (their recorded traffic stays valid while these hold).
HARD_SOURCES = ("ecc_hard.cu", "ecc_internal.cuh", "ecc_keys.cuh")


def _code_only(text: str) -> str:
    """The source without comments and blank lines (a comment edit leaves the kernels as they
    were, so it does not void their recorded counters)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(ln.rstrip() for ln in text.splitlines() if ln.strip())


def kernel_source_hash(files=HARD_SOURCES):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "euler_characteristic_curves_gb300", "csrc")
    for f in sorted(files):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode())
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if it matches the current source."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        d = json.load(fh)
    ent = d.get(kernel_key)
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent.get("bytes_per_launch")


class NvmlClockSampler:
    """Reads SM clocks, power and clock-event reasons through NVML (read-only queries, loaded
    with ctypes) every 2 ms while the timed region runs; a short timed region still gets many
    samples. Raises OSError when NVML cannot be loaded (the nvidia-smi sampler is used then)."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int, period_s: float = 0.002):
        import ctypes

        import torch

        self.ct = ctypes
        self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
        if self.nvml.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        props = torch.cuda.get_device_properties(device_index)
        bus = getattr(props, "pci_bus_id", None)
        dom = getattr(props, "pci_domain_id", 0)
        dev = getattr(props, "pci_device_id", 0)
        self.handle = ctypes.c_void_p()
        ok = False
        if bus is not None:
            pci = f"{dom:08x}:{bus:02x}:{dev:02x}.0".encode()
            ok = self.nvml.nvmlDeviceGetHandleByPciBusId_v2(pci, ctypes.byref(self.handle)) == 0
        if not ok and self.nvml.nvmlDeviceGetHandleByIndex_v2(
                ctypes.c_uint(device_index), ctypes.byref(self.handle)) != 0:
            raise OSError("no NVML handle for the device")
        self.reasons_fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        self.period = period_s
        self.samples = []
        self.stop_flag = False
        self.thread = None

    def _one(self):
        ct = self.ct
        sm, smax, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ct.byref(sm)) != 0:  # SM clock
            return None
        self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ct.byref(smax))
        self.nvml.nvmlDeviceGetPowerUsage(self.handle, ct.byref(mw))
        self.reasons_fn(self.handle, ct.byref(rs))
        return sm.value, smax.value, mw.value / 1000.0, rs.value

    def start(self):
        import threading
        import time

        def run():
            while not self.stop_flag:
                s = self._one()
                if s is not None:
                    self.samples.append(s)
                time.sleep(self.period)

        self.thread = threading.Thread(target=run, daemon=True)
        self.thread.start()

    def stop(self):
        self.stop_flag = True
        if self.thread:
            self.thread.join(timeout=5)
        s = self._one()  # at least one sample, taken at the end of the timed region
        if s is not None:
            self.samples.append(s)
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        reasons = sorted({name for *_, r in self.samples for bit, name in self.REASONS.items()
                          if r & bit})
        return {"sm_mhz": statistics.median(x[0] for x in self.samples),
                "sm_max_mhz": max(x[1] for x in self.samples), "samples": len(self.samples),
                "power_w_max": max(x[2] for x in self.samples), "reasons": reasons,
                "sampler": "NVML every 2 ms"}


def clock_sampler(device_index: int):
    """NVML sampler when NVML loads, else the nvidia-smi one."""
    try:
        return NvmlClockSampler(device_index)
    except (OSError, AttributeError):
        return ClockSampler(device_index)


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "samples": len(sm), "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons)}


# Soft-path roofline. The soft kernels evaluate one sigmoid term per (listed voxel, threshold)
# in the forward pass and again in the backward pass. A term takes one special-function (XU)
# operation -- the reciprocal of 1 + e, with e = E_p F_k a plain product -- or two on tiles whose
# exponents leave the factorised range (ex2 + reciprocal), plus about 4 FP32 operations forward
# (E F, 1 + e, the select, the accumulate) and 7 backward (also w = r - r^2 and the two
# accumulations of c w and g w). GB300 issues 16 XU and 128 FP32 operations per clock per SM on
# 152 SMs, so at one XU operation per term the XU pipe bounds the rate:
#     peak terms/s = 152 * 16 * f_sm.
SM_COUNT, XU_PER_CLK, FP32_PER_CLK = 152, 16, 128
FP32_PER_TERM = (4 + 7) / 2  # average over the forward and the backward term


def soft_roofline(p, ms, stats, clocks):
    n_list, n_direct, n_tiles = stats
    K = p[3]
    terms = 2 * n_list * K  # forward + backward
    xu_ops = terms * (1.0 + (n_direct / n_tiles if n_tiles else 0.0))
    f_sm = (clocks.get("sm_max_mhz") or 2070.0) * 1e6
    xu_peak = SM_COUNT * XU_PER_CLK * f_sm
    fp32_peak = SM_COUNT * FP32_PER_CLK * f_sm
    achieved = terms / (ms * 1e-3)
    return {"listed_voxels": n_list, "direct_tiles": n_direct, "tiles": n_tiles,
            "dense_terms": 2 * part_voxels(p) * K * part_dirs(p),
            "roofline": {"bound": "xu", "unit": "Gterms/s",
                         "achieved": round(achieved / 1e9, 2),
                         "peak": round(xu_peak / 1e9, 2),
                         "frac": round(xu_ops / (ms * 1e-3) / xu_peak, 4),
                         "fp32_frac": round(terms * FP32_PER_TERM / (ms * 1e-3) / fp32_peak, 4),
                         "peak_source": "derived: 152 SMs x 16 XU ops/clk x max SM clock, one "
                                        "XU op per term (two on direct-form tiles)",
                         "timing": "CUDA events around forward + backward library calls"}}


# ------------------------------------------------------------------------------------ our arm

def make_inputs(parts, device):
    import numpy as np
    import torch

    from euler_characteristic_curves_gb300 import synthetic

    inputs = []
    rank, world, _ = dist_env()
    for p in parts:
        if p[0] == "shard":  # this rank's slab of the volume (the whole volume at N = 1)
            from euler_characteristic_curves_gb300 import shard

            _, shape, batch, kind, nbins, vmin, vmax, seed = p[:8]
            vol = synthetic.grf(shape, seed, device=device)
            a, b = shard.slab_plan(shape[0], world)[rank]
            slab = vol[a:b + 1].clone()
            del vol
            torch.cuda.empty_cache()
            inputs.append({"img": slab, "ndim": 3, "rank": rank, "planes": (a, b)})
            continue
        if p[0] == "hard":
            _, shape, batch, kind, nbins, vmin, vmax, seed = p[:8]
            if part_slab(p):
                img = synthetic.grf(shape, seed, device=device)
                inputs.append({"host": img.cpu().pin_memory(), "ndim": len(shape)})
                del img
                continue
            if kind == "u8blur":
                img = torch.from_numpy(synthetic.blurred_noise_u8(shape, seed)).to(device)
            elif kind == "u8grf":
                img = synthetic.quantise_u8(synthetic.grf(shape, seed, device=device))
            else:
                img = synthetic.grf(shape, seed, device=device,
                                    batch=batch if batch > 1 else None)
            if batch == 1:
                img = img.unsqueeze(0)
            inputs.append({"img": img.contiguous(), "ndim": len(shape)})
        else:
            _, shape, batch, K, lam, s_img, s_u, s_g = p[:8]
            nd = part_dirs(p)
            img = synthetic.grf(shape, s_img, device=device, batch=batch)
            tau = torch.from_numpy(synthetic.uniform_thresholds(K)).to(device)
            if nd == 1:
                u = torch.from_numpy(synthetic.soft_direction(len(shape), s_u)).to(device)
                g = torch.from_numpy(synthetic.upstream_grad((batch, K), s_g)).to(device)
            else:
                u = torch.from_numpy(np.stack([synthetic.soft_direction(len(shape), s_u + j)
                                               for j in range(nd)])).to(device)
                g = torch.from_numpy(synthetic.upstream_grad((batch, nd, K), s_g)).to(device)
            alpha = torch.ones(1, dtype=torch.float32, device=device)
            inputs.append({"img": img.contiguous(), "tau": tau, "u": u, "g": g, "alpha": alpha,
                           "lam": lam})
    torch.cuda.synchronize()
    return inputs


def hard_launches(p, sms):
    """Kernels one hard-ECC call launches: a 3-D call the pass and the scan; a 2-D call the pass
    alone (an image's only block stores its curve, several blocks add the running sums of their
    histograms)."""
    if part_slab(p):  # slabs sharing one plane: a 3-D pass each, a plane pass from the second
        D, S, n, a = p[1][0], part_slab(p), 0, 0  # slab on, and one scan at the end
        while True:
            b = min(a + S - 1, D - 1)
            n += 1
            if b == D - 1:
                return 2 * n
            a = b
    if len(p[1]) != 2:
        return 2
    return 1  # a 2-D image's blocks add the running sums of their histograms: no scan launch


class OurStep:
    """One pass of the hot path through the library's public binding (device-resident)."""

    def __init__(self, parts, inputs, device):
        import torch

        from euler_characteristic_curves_gb300 import ecc

        self.ecc = ecc
        self.parts, self.inputs = parts, inputs
        self.outs = []
        for p, x in zip(parts, inputs):
            if p[0] == "shard":
                self.outs.append(torch.empty(p[4], dtype=torch.int64, device=device))
            elif p[0] == "hard" and part_slab(p):
                nbytes = ecc.hard_stream_buffer_bytes(p[1], torch.float32, part_slab(p))
                self.outs.append({"out": torch.empty(p[4], dtype=torch.int64, device=device),
                                  "buf": torch.empty(nbytes, dtype=torch.uint8, device=device)})
            elif p[0] == "hard":
                self.outs.append(torch.empty((x["img"].shape[0], p[4]), dtype=torch.int64,
                                             device=device))
            else:
                K = p[3]
                nb = x["img"].shape[0]
                nd = part_dirs(p)
                ws = torch.empty(ecc.soft_workspace_bytes(p[1], nb, K, nd), dtype=torch.uint8,
                                 device=device)
                s = torch.empty((nb, nd, K) if nd > 1 else (nb, K), dtype=torch.float32,
                                device=device)
                self.outs.append({"ws": ws, "s": s})
        sms = torch.cuda.get_device_properties(device).multi_processor_count
        self.launches_per_step = sum(
            hard_launches(p, sms) if p[0] == "hard" else
            (2 + (x["rank"] > 0)) if p[0] == "shard" else 6 for p, x in zip(parts, inputs))

    def run_part(self, i):
        p, x, o = self.parts[i], self.inputs[i], self.outs[i]
        if p[0] == "shard":
            from euler_characteristic_curves_gb300 import shard

            o.zero_()
            shard.volume_partial(x["img"], p[4], p[5], p[6], x["rank"], o)
            shard._default_allreduce(None)(o)
            self.ecc.hist_to_curve(o)
        elif p[0] == "hard" and part_slab(p):
            self.ecc.ecc_hard_stream(x["host"], p[4], p[5], p[6], slab_planes=part_slab(p),
                                     buf=o["buf"], out=o["out"])
        elif p[0] == "hard":
            self.ecc.ecc_hard(x["img"], p[4], p[5], p[6], ndim=x["ndim"], out=o)
        elif part_dirs(p) == 1:
            self.ecc.ecc_soft_fwd(x["img"], x["tau"], x["lam"], x["alpha"], x["u"], ws=o["ws"],
                                  out=o["s"])
            o["grads"] = self.ecc.ecc_soft_bwd(x["img"], x["tau"], x["lam"], x["alpha"], x["u"],
                                               x["g"], o["ws"])
        else:
            self.ecc.ecc_soft_ect_fwd(x["img"], x["tau"], x["lam"], x["alpha"], x["u"],
                                      ws=o["ws"], out=o["s"], ndim=len(p[1]))
            o["grads"] = self.ecc.ecc_soft_ect_bwd(x["img"], x["tau"], x["lam"], x["alpha"],
                                                   x["u"], x["g"], o["ws"], ndim=len(p[1]))

    def link_peaks(self):
        """Per streamed part: the host-to-device copy rate of its whole host volume in one
        cudaMemcpyAsync (GB/s), the ceiling of the streamed path."""
        import torch

        out = {}
        for p, x, o in zip(self.parts, self.inputs, self.outs):
            if p[0] == "hard" and part_slab(p):
                h = x["host"]
                d = torch.empty(h.shape, dtype=h.dtype, device=o["out"].device)
                d.copy_(h, non_blocking=True)
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(3):
                    d.copy_(h, non_blocking=True)
                e1.record()
                torch.cuda.synchronize()
                ms = e0.elapsed_time(e1) / 3
                out[part_name(p)] = round(h.numel() * h.element_size() / (ms * 1e-3) / 1e9, 1)
                del d
        return out

    def soft_stats(self):
        """Per soft part: [listed voxels, direct-form tiles, tiles] of the last forward pass."""
        out = {}
        for p, x, o in zip(self.parts, self.inputs, self.outs):
            if p[0] == "soft":
                st = self.ecc.ecc_soft_ect_stats(x["img"], p[3], part_dirs(p), o["ws"],
                                                 ndim=len(p[1]))
                out[part_name(p)] = [int(v) for v in st.cpu().tolist()]
        return out

    def results_of(self, i):
        p, o = self.parts[i], self.outs[i]
        if p[0] == "shard":
            return [o]
        if p[0] == "hard":
            return [o["out"] if part_slab(p) else o]
        return [o["s"], *o["grads"].values()]

    def results(self):
        return [t for i in range(len(self.parts)) for t in self.results_of(i)]


def capture_parts(step, parts, device):
    """Captures each part's library calls into its own CUDA graph and returns a runner that
    replays part i. Every replay launches all of the part's kernels again; what it removes is the
    host's per-call work (argument checks, ctypes, launch submission), which for small parts
    takes longer than the GPU work and leaves the GPU idle between calls. Before returning it
    checks that a replay gives the same bits as an eager call of the same part."""
    import torch

    if any(part_slab(p) for p in parts):
        raise SystemExit("--graph: the streamed part copies from host memory with its own "
                         "streams and is not captured")
    graphs, captured = [], []
    for i in range(len(parts)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step.run_part(i)
        graphs.append(g)
        o = step.outs[i]
        captured.append(dict(o["grads"]) if isinstance(o, dict) and "grads" in o else None)
    for i, g in enumerate(graphs):
        g.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in step.results_of(i)]
        step.run_part(i)
        torch.cuda.synchronize()
        want = step.results_of(i)
        if len(got) != len(want) or not all(torch.equal(a, b) for a, b in zip(got, want)):
            raise SystemExit(f"--graph: replay of part {part_name(parts[i])} differs from the "
                             "eager call")
        if captured[i] is not None:  # the eager call made new gradient tensors
            step.outs[i]["grads"] = captured[i]
    return lambda i: graphs[i].replay()


def time_ours(args, parts, rank, world, device):
    import torch

    inputs = make_inputs(parts, device)
    step = OurStep(parts, inputs, device)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        for i in range(len(parts)):
            step.run_part(i)
    torch.cuda.synchronize()
    barrier(world)
    sampler = clock_sampler(torch.cuda.current_device())
    sampler.start()
    run = step.run_part
    if args.graph:
        run = capture_parts(step, parts, device)
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in parts] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(world)
    start.record(stream)
    for s in range(args.steps):
        for i in range(len(parts)):
            ev[s][i][0].record(stream)
            run(i)
            ev[s][i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    total_ms = start.elapsed_time(end)
    part_ms = [statistics.mean(ev[s][i][0].elapsed_time(ev[s][i][1]) for s in range(args.steps))
               for i in range(len(parts))]
    total_ms = max_over_ranks(total_ms, world)
    soft_stats = step.soft_stats()
    soft_stats["_link_peaks"] = step.link_peaks()
    e2e = None if args.no_e2e else time_e2e(args, parts, inputs, step, device, world)
    return total_ms, part_ms, clocks, step.launches_per_step * args.steps, e2e, soft_stats


def time_e2e(args, parts, inputs, step, device, world):
    """Same step through the public binding with HOST inputs: every step copies its inputs from
    pinned host memory to the device and reads the results back. A single 3-D volume goes through
    the library's host-input call (ecc_hard_stream), which overlaps its slab copies with the slab
    kernels; the other parts copy and run on a second stream beside it."""
    import torch

    host = []
    h2d = 0
    streamed = {}  # part index -> (host volume, slab buffer, output row) for 3-D volumes
    for i, (p, x) in enumerate(zip(parts, inputs)):
        hx = {}
        for k, v in x.items():
            if isinstance(v, torch.Tensor) and not v.is_cuda:
                # a streamed volume already lives in host memory: the call copies it itself
                h2d += v.numel() * v.element_size()
            elif isinstance(v, torch.Tensor):
                hv = torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
                hv.copy_(v)
                hx[k] = hv
                h2d += v.numel() * v.element_size()
        if p[0] == "hard" and not part_slab(p) and len(p[1]) == 3 and p[2] == 1:
            vol = hx.pop("img")[0]
            nbytes = step.ecc.hard_stream_buffer_bytes(p[1], vol.dtype, E2E_SLAB)
            buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
            streamed[i] = (vol, buf, step.outs[i][0])
        host.append(hx)
    res_dev = step.results()
    d2h = sum(t.numel() * t.element_size() for t in res_dev)
    res_host = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in res_dev]
    steps = max(1, min(args.steps, 8))
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream(device=device)

    def one():
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for i, (hx, x) in enumerate(zip(host, inputs)):
                if i in streamed:
                    continue
                for k, hv in hx.items():
                    x[k].copy_(hv, non_blocking=True)
                step.run_part(i)
        for i, (vol, buf, out) in streamed.items():
            p = parts[i]
            step.ecc.ecc_hard_stream(vol, p[4], p[5], p[6], slab_planes=E2E_SLAB, buf=buf,
                                     out=out, stream=stream)
        stream.wait_stream(side)
        for hr, t in zip(res_host, step.results()):
            hr.copy_(t, non_blocking=True)

    link = host_link_gbs(device)
    for _ in range(max(1, args.warmup)):  # the same warm-up count as the device-side timing
        one()
    torch.cuda.synchronize()
    barrier(world)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    marks[0].record(stream)
    for i in range(steps):
        one()
        marks[i + 1].record(stream)
    torch.cuda.synchronize()
    per_step = [marks[i].elapsed_time(marks[i + 1]) for i in range(steps)]
    ms = max_over_ranks(marks[0].elapsed_time(marks[-1]) / steps, world)
    med = max_over_ranks(statistics.median(per_step), world)
    hard_vox = sum(part_voxels(p) for p in parts if p[0] in ("hard", "shard")) or \
        sum(part_voxels(p) for p in parts)
    ranks = 1 if any(p[0] == "shard" for p in parts) else world  # a sharded volume: one problem
    return {"value": round(hard_vox * ranks / (ms * 1e-3) / 1e9, 3), "unit": "Gvoxels/s",
            "ms_per_step": round(ms, 3), "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": steps,
            "link_gbs": link, "link_floor_ms": round(h2d / (link * 1e9) * 1e3, 3),
            "ms_per_step_median": round(med, 3),
            "value_median": round(hard_vox * ranks / (med * 1e-3) / 1e9, 3),
            "ms_steps": [round(x, 2) for x in per_step],
            "path": ("3-D volumes through ecc_hard_stream from pinned host memory in "
                     f"{E2E_SLAB}-plane slabs; other parts copied and run on a second stream"
                     if streamed else "inputs copied from pinned host memory, then the step")}


E2E_SLAB = 64  # planes per slab of a 3-D volume in the end-to-end timing


def host_link_gbs(device, nbytes=1 << 30):
    """Host-to-device copy rate of this machine (GB/s): one pinned buffer copied three times. The
    end-to-end step cannot beat its input bytes at this rate; it varies between boxes."""
    import torch

    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device=device)
    d.copy_(h, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(3):
        d.copy_(h, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / 3
    del h, d
    return round(nbytes / (ms * 1e-3) / 1e9, 1)


# ------------------------------------------------------------------------------------ oracle arm

SAMPLE_2D = 512           # 2-D parts: a 512 x 512 crop of one image
SAMPLE_3D = (32, 128, 128)  # 3-D parts: a 32 x 128 x 128 crop
SAMPLE_SOFT = 128        # soft part: one 128 x 128 image, all K thresholds, fwd + bwd
SAMPLE_SOFT_3D = 24      # 3-D soft part: one 24^3 volume
SAMPLE_ECT = 48          # transform part: one 48^2 image, all directions
SAMPLE_TEXT = ("each 2-D part cropped to 512^2 (one image), each 3-D part to 32x128x128, "
               "a 2-D soft part one 128^2 image (a 3-D one a 24^3 volume, a transform part one "
               "48^2 image with all directions) with all K thresholds (fwd + bwd)")


def oracle_sample_step(parts, cache):
    """The oracle on a bounded sample of every part of the workload; returns voxels processed."""
    import oracle
    from euler_characteristic_curves_gb300 import synthetic

    import numpy as np

    vox = 0
    for p in parts:
        key = part_name(p)
        if key not in cache:
            if p[0] in ("hard", "shard"):
                _, shape, batch, kind, nbins, vmin, vmax, seed = p[:8]
                if len(shape) == 2:
                    sh = (min(shape[0], SAMPLE_2D), min(shape[1], SAMPLE_2D))
                else:
                    sh = tuple(min(a, b) for a, b in zip(shape, SAMPLE_3D))
                if kind == "u8blur":
                    img = synthetic.blurred_noise_u8(sh, seed)
                elif kind == "u8grf":
                    img = synthetic.quantise_u8(synthetic.grf(sh, seed))
                else:
                    img = synthetic.grf(sh, seed)
                cache[key] = img
            else:
                _, shape, batch, K, lam, s_img, s_u, s_g = p[:8]
                nd = part_dirs(p)
                if nd > 1:
                    sh = tuple(min(a, SAMPLE_ECT) for a in shape)
                elif len(shape) == 2:
                    sh = (min(shape[0], SAMPLE_SOFT), min(shape[1], SAMPLE_SOFT))
                else:
                    sh = tuple(min(a, SAMPLE_SOFT_3D) for a in shape)
                U = np.stack([synthetic.soft_direction(len(shape), s_u + j) for j in range(nd)])
                cache[key] = (synthetic.grf(sh, s_img), synthetic.uniform_thresholds(K), U,
                              synthetic.upstream_grad((1, nd, K), s_g))
        x = cache[key]
        if p[0] in ("hard", "shard"):
            oracle.ecc_hard(x, p[4], p[5], p[6])
            vox += x.size
        else:
            img, tau, U, g = x
            oracle.ecc_soft_ect_fwd(img, tau, p[4], 1.0, U)
            oracle.ecc_soft_ect_bwd(img, tau, p[4], 1.0, U, g[0], want_img=False)
            vox += img.size
    return vox


def time_oracle(steps, warmup, parts, min_seconds=0.0):
    """Times `steps` sample passes (after `warmup`), continuing until min_seconds have passed."""
    cache = {}
    for _ in range(warmup):
        oracle_sample_step(parts, cache)
    t0 = time.perf_counter()
    vox, n = 0, 0
    while n < steps or time.perf_counter() - t0 < min_seconds:
        vox += oracle_sample_step(parts, cache)
        n += 1
    dt = time.perf_counter() - t0
    return vox, dt, n


def _oracle_worker(task):
    parts, min_seconds = task
    vox, dt, _ = time_oracle(1, 1, parts, min_seconds)
    return vox, dt


def time_oracle_all_cores(parts, min_seconds):
    """The same plain oracle in one process per host core, each on its own copy of the sample
    (independent problems); returns the summed rate (voxels/s) and the number of processes.
    Workers start with 'spawn', so the parent's CUDA context is not inherited."""
    import multiprocessing as mp

    import oracle

    from concurrent.futures import ProcessPoolExecutor

    oracle.build()  # compile once before the workers load it
    n = max(1, min(os.cpu_count() or 1, 64))
    with ProcessPoolExecutor(n, mp_context=mp.get_context("spawn")) as ex:
        futs = [ex.submit(_oracle_worker, (parts, min_seconds)) for _ in range(n)]
        res = [f.result(timeout=300.0 + 4.0 * min_seconds) for f in futs]
    return sum(v / dt for v, dt in res), n


# ------------------------------------------------------------------------------------ dist

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world, backend):
    if world > 1:
        import torch.distributed as dist

        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Slowest rank's value (timings are maxima over ranks)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------ main

def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="headline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end timing (for profiler launch lists of the step)")
    ap.add_argument("--graph", action="store_true",
                    help="time replays of one CUDA graph per part (the same library calls, "
                         "captured once) instead of eager calls")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local = dist_env()
    parts = WORKLOADS[args.workload]
    hard_vox = sum(part_voxels(p) for p in parts if p[0] in ("hard", "shard"))
    unit_vox = hard_vox if hard_vox else sum(part_voxels(p) for p in parts)
    # a sharded volume is one problem split over the ranks (total work fixed as N grows)
    strong = any(p[0] == "shard" for p in parts)
    config = {"workload": DESCRIPTION.get(args.workload, args.workload),
              "parts": [part_name(p) for p in parts],
              "l2": "inputs larger than L2 (the 268 MB image and the 4 GiB volume evict L2 "
                    "between passes)" if args.workload == "headline" else "not flushed",
              "parallelism": (f"one volume in {world} slabs sharing a plane, one all-reduce"
                              if strong else f"independent replicas x{world}"),
              "timing": ("one CUDA graph per part (its library calls captured once), replayed "
                         "every step" if args.graph else "eager library calls")}

    if args.impl == "reference":
        if rank != 0:
            return 0
        config["timing"] = "the oracle on one host core, a bounded sample of every part per step"
        vox, dt, _ = time_oracle(args.steps, args.warmup, parts)
        value = vox / dt / 1e9
        line = {"impl": "reference", "metric": METRIC, "value": round(value, 6),
                "unit": "Gvoxels/s", "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
                "higher_is_better": True, "scaling": "strong" if strong else "weak",
                "vs_baseline": None,
                "dtype": "f64 oracle on f32/u8 inputs", "data": "synthetic (seeded GRF)",
                "config": config,
                "cpu_baseline": {"value": round(value, 6), "unit": "Gvoxels/s", "cores": 1,
                                 "kind": "oracle", "sample": "per step: " + SAMPLE_TEXT},
                "e2e": {"value": round(value, 6), "unit": "Gvoxels/s",
                        "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    import torch

    init_dist(world, "nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    from euler_characteristic_curves_gb300 import build as libbuild

    libbuild.build()
    total_ms, part_ms, clocks, launches, e2e, soft_stats = time_ours(args, parts, rank, world,
                                                                     device)
    ms_step = total_ms / args.steps
    value = unit_vox * (1 if strong else world) / (ms_step * 1e-3) / 1e9

    peak, peak_kind = load_peaks()
    # dominant kernel: the part with the largest device time
    dom = max(range(len(parts)), key=lambda i: part_ms[i])
    breakdown = {}
    for i, p in enumerate(parts):
        ms = part_ms[i]
        ent = {"ms": round(ms, 4), "gvoxels_s": round(part_voxels(p) / (ms * 1e-3) / 1e9, 3)}
        if p[0] in ("hard", "shard"):
            alg = part_alg_bytes(p, time_inputs_planes(p, rank, world))
            ent["hbm_gbs"] = round(alg / (ms * 1e-3) / 1e9, 1)
            if part_slab(p):  # streamed: every voxel crosses the host link once per step
                ent["link_gbs"] = ent["hbm_gbs"]
                lp = soft_stats["_link_peaks"].get(part_name(p))
                if lp:
                    ent["link_peak_gbs"] = lp  # one plain copy of the host volume, measured
                    ent["link_frac"] = round(ent["link_gbs"] / lp, 4)
            ent["hbm_frac"] = round(alg / (ms * 1e-3) / 1e9 / peak, 4)
        if p[0] == "soft":
            ent.update(soft_roofline(p, ms, soft_stats[part_name(p)], clocks))
        breakdown[part_name(p)] = ent
    roofline = None
    pd = parts[dom]
    if pd[0] in ("hard", "shard"):
        alg = part_alg_bytes(pd, time_inputs_planes(pd, rank, world))
        achieved = alg / (part_ms[dom] * 1e-3) / 1e9
        key = hard_kernel_name(pd)
        roofline = {"bound": "hbm", "kernel": key, "achieved": round(achieved, 1),
                    "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                    "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                    "traffic": recorded_traffic(f"{key}:{part_name(pd)}"),
                    "algorithmic_bytes": int(alg),
                    "timing": "CUDA events around the library call (memset + kernel + scan)"}

    cpu = cpu_all = None
    if rank == 0 and not args.no_cpu_baseline:
        vox, dt, npass = time_oracle(1, 1, parts, min_seconds=10.0)
        cpu = {"value": round(vox / dt / 1e9, 6), "unit": "Gvoxels/s", "cores": 1,
               "kind": "oracle", "seconds": round(dt, 2),
               "sample": f"{npass} passes (single-threaded C, ~10 s), each: " + SAMPLE_TEXT}
        rate, workers = time_oracle_all_cores(parts, 10.0)
        cpu_all = {"value": round(rate / 1e9, 6), "unit": "Gvoxels/s", "cores": workers,
                   "kind": "oracle",
                   "sample": f"one process per core, each ~10 s of passes over: " + SAMPLE_TEXT}
    soft_ms = [part_ms[i] for i, p in enumerate(parts) if p[0] == "soft"]
    line = {"metric": METRIC, "value": round(value, 3), "unit": "Gvoxels/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "strong" if strong else "weak",
            "vs_baseline": None,
            "dtype": "f32 compare / int32+int64 histogram (hard); f32 + fp64 reductions (soft)",
            "data": "synthetic (seeded Gaussian random fields, k^-3 spectrum)",
            "config": config, "parts": breakdown,
            "soft_fwd_bwd_ms": round(soft_ms[0], 4) if soft_ms else None,
            "soft_roofline": next((breakdown[part_name(p)]["roofline"] for p in parts
                                   if p[0] == "soft"), None),
            "roofline": roofline, "cpu_baseline": cpu, "cpu_baseline_all_cores": cpu_all,
            "e2e": e2e,
            "gpu_launches": launches, "clocks": clocks,
            "kernel_source": kernel_source_hash()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
