#!/usr/bin/env python
"""Benchmark of the multiresolution hash-grid encoding on one B300 per rank.

A step is one full pass of the hot path over one batch of synthetic points:
zero the gradient table, Hermite forward (gamma, grad gamma, Laplacian of
every point and level) and Hermite backward (scatter of the coefficient
gradients).  The default workload is the 3D Hermite grid: N = 2^21 points in
[0,1]^3, L = 16 levels from N_min = 16 to N_max = 512, F = 2, 2^19 entries
per order table (packed layout), fp32 coefficients U[-1e-2, 1e-2], N(0,1)
upstream gradients.  ``--config`` picks another of the five workloads.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
a bounded sample of the same workload instead (the oracle is a deliberately
slow fp64 program; the ratio against it is context, not a target).

``--siren`` times the encoder with its consumer instead: Hermite forward,
the SIREN chain rule (u, grad u, lap u from gamma, grad gamma, lap gamma),
the SIREN's backward from N(0,1) gradients of u, grad u and lap u, and the
Hermite backward of the SIREN's input gradients.

Multi-GPU (torchrun): every rank runs its own replica on its own shard of
points (the forward and backward of different points are independent); the
timed region is bracketed by barriers and the slowest rank's time is used.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "encoded points/s (Hermite fwd γ,∇γ,∇²γ + bwd) at 1 B300; % of L2/HBM gather roofline"
METRIC_FD = ("encoded points/s (INGP-FD: d-linear encodes at x and the 2d stencil points x +- eps e_i, + bwd) "
             "at 1 B300; % of L2 gather roofline")
METRIC_RBF = ("encoded points/s (Gaussian-RBF grid fwd gamma, grad, Laplacian + bwd) at 1 B300; "
              "% of the measured ceiling")
METRIC_HESSIAN = "encoded points/s (Hermite fwd γ,∇γ, full Hessian + bwd) at 1 B300; % of L2 gather roofline"
METRIC_SIREN = ("points/s of encoder + SIREN (Hermite fwd γ,∇γ,∇²γ; SIREN u,∇u,∇²u; SIREN bwd; Hermite bwd) "
                "at 1 B300; % of the dominant kernel's roofline")
L2_BYTES = 126 * 1024 * 1024
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")


def parse_args():
    p = argparse.ArgumentParser(description=__doc__)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--config", type=int, default=4,
                   help="workload 1..10 (default 4: 3D Hermite, 2^21 points; 10: workload 3 in shuffled order)")
    p.add_argument("--level-mask", type=lambda s: int(s, 0), default=None)
    p.add_argument("--layout", choices=["feature", "point"], default="feature")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-all-configs", action="store_true",
                   help="skip the other workloads reported beside the headline (workloads 1, 2, 3, 3 shuffled, "
                        "5 at L_active 4/10/16)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-sample", type=int, default=1 << 20, help="points in the oracle's timed sample")
    p.add_argument("--points", type=int, default=None, help="override the workload's point count (profiling)")
    p.add_argument("--hessian", action="store_true",
                   help="Hermite workloads: the full-Hessian entry points (every d2/dx_i dx_j) instead of the "
                        "Laplacian ones")
    p.add_argument("--siren", action="store_true",
                   help="Hermite workloads: time the encoder with its SIREN chain-rule consumer (forward and "
                        "backward of both)")
    p.add_argument("--probe-patterns", action="store_true",
                   help="print the L2 random-row gather / RED rates for 1, 2 and 4 lanes per row "
                        "(32- and 64-byte rows) as one JSON line, then exit")
    p.add_argument("--record-traffic", metavar="NCU_LOG", default=None,
                   help="parse an ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum log of the benchmark "
                        "command and record per-launch DRAM traffic (with the kernel-source hash) in "
                        "profiles/dram_traffic.json, then exit")
    p.add_argument("--record-traffic-kernel", choices=["fwd", "bwd"], default="fwd",
                   help="which kernel the --record-traffic capture covered (one kernel per capture)")
    return p.parse_args()


# ---------------------------------------------------------------------------
# DRAM traffic recorded from an ncu capture, valid while the kernels are unchanged
# ---------------------------------------------------------------------------

# Sources of kernels whose DRAM traffic is not recorded: the roofline probes, the SIREN consumer and
# the other encodings (d-linear, INGP-FD, Gaussian-RBF) -- a change there leaves the Hermite kernels'
# recorded traffic valid.
UNRECORDED_SOURCES = ("probes.cu", "hg_probe.h", "siren.cu", "siren_tc.cuh", "linear.cu", "linear_fd.cu", "rbf.cu")


def kernel_source_hash() -> str:
    """sha256 over the sources of the Hermite encoding kernels, their launch
    code and the headers they include (UNRECORDED_SOURCES left out)."""
    import glob
    import hashlib
    h = hashlib.sha256()
    pkg = os.path.join(ROOT, "multiresolution_hash_grid_02_b300", "csrc")
    files = sorted(f for f in glob.glob(os.path.join(pkg, "*.cu")) + glob.glob(os.path.join(pkg, "*.cuh")) +
                   glob.glob(os.path.join(pkg, "*.h")) + glob.glob(os.path.join(ROOT, "include", "*.h"))
                   if os.path.basename(f) not in UNRECORDED_SOURCES)
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def parse_ncu_dram_log(path: str) -> dict:
    """{kernel name: {"dram_read": B, "dram_write": B, "launches": k}} from ncu's
    default text output (units Kbyte/Mbyte/Gbyte are decimal)."""
    import re
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "Tbyte": 1e12}
    out, cur = {}, None
    with open(path) as f:
        for line in f:
            m = re.match(r"\s{2}(\S.*?)\s+\(\d+, \d+, \d+\)x\(\d+, \d+, \d+\)", line)
            if m:
                base = m.group(1).split("(")[0]
                k = re.search(r"(\w+_kernel\b.*)$", base)
                cur = (k.group(1) if k else base).strip()
                out.setdefault(cur, {"dram_read": 0.0, "dram_write": 0.0, "launches": 0})
                out[cur]["launches"] += 1
                continue
            m = re.match(r"\s+dram__bytes_(read|write)\.sum\s+(\S+)\s+([\d.,]+)", line)
            if m and cur:
                out[cur]["dram_" + m.group(1)] += float(m.group(3).replace(",", "")) * scale[m.group(2)]
    for k, v in out.items():
        n = max(1, v["launches"])
        v["bytes_per_launch"] = (v["dram_read"] + v["dram_write"]) / n
    return out


def record_traffic(log_path: str, workload: str, command: str):
    """Store the per-launch DRAM traffic of one bench configuration (key
    `workload`) beside those of the others captured from the same kernel
    sources; a capture from changed sources starts the file afresh."""
    sha = kernel_source_hash()
    try:
        with open(TRAFFIC_FILE) as f:
            data = json.load(f)
    except (OSError, ValueError):
        data = {}
    if data.get("source_sha256") != sha or "entries" not in data:
        data = {"source_sha256": sha, "entries": {}}
    # one capture per kernel (forward, backward): each adds its kernels to the configuration's entry
    entry = data["entries"].setdefault(workload, {"commands": [], "kernels": {}})
    entry.pop("command", None)
    entry.setdefault("commands", [])
    if command not in entry["commands"]:
        entry["commands"].append(command)
    entry.setdefault("kernels", {}).update(parse_ncu_dram_log(log_path))
    os.makedirs(os.path.dirname(TRAFFIC_FILE), exist_ok=True)
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(data, f, indent=1)
    print(json.dumps(data["entries"][workload]))


def recorded_traffic(workload: str, kernel_prefix: str):
    """Per-launch DRAM bytes of the kernel from the recorded capture, or None
    when there is none for this configuration or the kernels changed since."""
    try:
        with open(TRAFFIC_FILE) as f:
            data = json.load(f)
    except (OSError, ValueError):
        return None
    if data.get("source_sha256") != kernel_source_hash():
        return None
    entry = data.get("entries", {}).get(workload)
    if not entry:
        return None
    for name, v in entry.get("kernels", {}).items():
        if name.startswith(kernel_prefix):
            return v["bytes_per_launch"]
    return None


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest value across ranks (the slowest rank's time); identity for
    one rank.  Uses the default process group (NCCL on GPUs, gloo on CPU)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# workload description and algorithmic byte counts
# ---------------------------------------------------------------------------

def describe(w, mask, layout, hessian=False, siren=False):
    res_note = f"N_min={w.n_min}, N_max={w.n_max}"
    lt = w.log2_T[0]
    return {
        "workload": w.name,
        "n_points": w.n_points,
        "d": w.d, "L": w.L, "F": w.F, "log2_T": lt, "n_min": w.n_min, "n_max": w.n_max,
        "table_dtype": w.dtype,
        "table_layout": "packed [L][T][2^d][F]" if w.kind == "hermite" else "[L][T][F]",
        "output_layout": layout + "-major",
        "active_levels": bin(mask).count("1"),
        "coords": w.coords,
        "description": f"{w.kind} d={w.d}: N={w.n_points} pts, L={w.L}, F={w.F}, T=2^{lt}, {res_note}, {w.dtype}",
        "l2_flush": "inputs larger than L2 (tables + upstream gradients + outputs exceed 126 MB per step)",
        "parallelism": "replicas",
        "second_order": ("full Hessian" if hessian else "Laplacian") if w.kind == "hermite" else None,
        **({"fd_eps": w.eps, "fd_outputs": "gamma(x) and the 2d stencil encodings (the network inputs of INGP-FD)"}
           if w.kind == "linear_fd" else {}),
        **({"rbf_eps_grid_units": w.eps, "rbf_rings": w.rings, "taps_per_point_level": (2 * w.rings) ** w.d}
           if w.kind == "rbf" else {}),
        **({"consumer": "SIREN u = W2 sin(omega (W1 gamma + b1)) + b2 with the chain rule for grad u and lap u",
            "siren_K": w.L * w.F, "siren_H": 64, "siren_O": 1, "siren_omega": 30.0} if siren else {}),
    }


def rbf_flops(w, mask):
    """Algorithmic FP32 flops of one RBF launch (forward or backward: the
    transposed contraction has the same count): the separable contraction's
    FMAs per (point, active level, feature) -- with K = 2 rings taps per
    axis, K (3K + 5) in 2D and K (K (3K + 5) + 6) in 3D -- times 2."""
    K = 2 * w.rings
    per = K * (3 * K + 5) if w.d == 2 else K * (K * (3 * K + 5) + 6)
    return 2 * per * w.F * w.n_points * bin(mask).count("1")


def siren_flops(n, d, K, H):
    """Algorithmic flops of the SIREN forward: its first layer contracts the
    d + 2 input rows of every point (gamma, d gamma/dx_i, lap gamma; K
    features) with W1 [H][K].  The backward's three contractions (the
    recomputed first layer, the input gradients and the W1 gradient) are
    three times that."""
    return 2 * n * (d + 2) * K * H


def fp32_peak_tflops(torch, sm_mhz: float) -> float:
    """FP32 FMA peak of the GPU: SMs x 128 lanes x 2 flops x SM clock."""
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return sms * 128 * 2 * sm_mhz * 1e6 / 1e12


def algorithmic_bytes(w, mask):
    """Per-launch algorithmic quantities (one launch covers all N points).

    fwd: compulsory coefficient bytes gathered = N * L_active * 2^d corners *
         (2^d slots * F * elem) for Hermite, N * L_active * 2^d * F * elem for
         d-linear.  INGP-FD counts the centre cell's rows only: a stencil
         point that stays in the cell needs no other row, so the compulsory
         set is at least those 2^d rows (crossing points add more).
    bwd: RED payload bytes = the same count of fp32 gradient values * 4 B.
    """
    La = bin(mask).count("1")
    es = 2 if w.dtype == "f16" else 4
    slots = (1 << w.d) if w.kind == "hermite" else 1
    taps = (2 * w.rings) ** w.d if w.kind == "rbf" else (1 << w.d)     # rbf: the ring box
    per_pt_level_vals = taps * slots * w.F
    gather = w.n_points * La * per_pt_level_vals * es
    red = w.n_points * La * per_pt_level_vals * 4
    return gather, red


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(rows), "reasons": reasons}


# ---------------------------------------------------------------------------
# the CPU oracle (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def metric_of(w, hessian=False, siren=False) -> str:
    if siren:
        return METRIC_SIREN
    if hessian:
        return METRIC_HESSIAN
    return {"linear_fd": METRIC_FD, "rbf": METRIC_RBF}.get(w.kind, METRIC)


def traffic_key(w, points=None, hessian=False):
    """Name under which the DRAM traffic of a bench configuration is recorded."""
    key = w.name if not points else f"{w.name}@{points}"
    return key + "+hessian" if hessian and w.kind == "hermite" else key


def add_hessian_upstream(w, inputs, rank=0):
    """Seeded upstream gradient of the full Hessian (point-major)."""
    from multiresolution_hash_grid_02_b300 import workloads as W
    inputs["g_hess"] = W.draw_upstream_hessian(np.random.default_rng(w.seed + 1000 + rank), w)


def oracle_setup(w, inputs):
    import oracle
    from multiresolution_hash_grid_02_b300 import workloads as W
    oracle.build()
    res = oracle.level_resolutions(w.L, w.n_min, w.n_max)
    if w.kind == "hermite":
        tabs = [np.ascontiguousarray(t, np.float64) for t in W.split_orders(inputs["table"], w.d)]
    else:
        tabs = np.ascontiguousarray(inputs["table"], np.float64)
    return oracle, res, tabs


def oracle_step(oracle, w, res, tabs, inputs, lo, hi, mask, threads, hessian=False):
    """Oracle forward + backward on points [lo, hi) of the workload."""
    x = inputs["coords"][lo:hi]
    if w.kind == "hermite" and hessian:
        oracle.encode_fwd_hessian(w.d, w.F, res, w.log2_T, tabs, x, level_mask=mask, nthreads=threads,
                                  with_mags=False)
        oracle.encode_bwd_hessian(w.d, w.F, res, w.log2_T, x, inputs["g_gamma"][lo:hi], inputs["g_dgamma"][lo:hi],
                                  inputs["g_hess"][lo:hi], level_mask=mask, with_mags=False, nthreads=threads)
    elif w.kind == "hermite":
        oracle.encode_fwd(w.d, w.F, res, w.log2_T, tabs, x, level_mask=mask, nthreads=threads, with_mags=False)
        oracle.encode_bwd(w.d, w.F, res, w.log2_T, x, inputs["g_gamma"][lo:hi], inputs["g_dgamma"][lo:hi],
                          inputs["g_lap"][lo:hi], level_mask=mask, with_mags=False, nthreads=threads)
    elif w.kind == "rbf":
        oracle.rbf_fwd(w.d, w.F, res, w.log2_T[0], tabs, x, w.eps, w.rings, level_mask=mask, nthreads=threads,
                       with_mags=False)
        oracle.rbf_bwd(w.d, w.F, res, w.log2_T[0], x, w.eps, w.rings, g_gamma=inputs["g_gamma"][lo:hi],
                       g_dgamma=inputs["g_dgamma"][lo:hi], g_lap=inputs["g_lap"][lo:hi], level_mask=mask,
                       with_mags=False, nthreads=threads)
    elif w.kind == "linear_fd":
        oracle.linear_fd_fwd(w.d, w.F, res, w.log2_T[0], tabs, x, w.eps, level_mask=mask, nthreads=threads,
                             with_mags=False)
        oracle.linear_fd_bwd(w.d, w.F, res, w.log2_T[0], x, w.eps, g_gamma=inputs["g_gamma"][lo:hi],
                             g_stencil=inputs["g_stencil"][lo:hi], level_mask=mask, with_mags=False,
                             nthreads=threads)
    else:
        oracle.linear_fwd(w.d, w.F, res, w.log2_T[0], tabs, x, level_mask=mask, nthreads=threads, with_mags=False)
        oracle.linear_bwd(w.d, w.F, res, w.log2_T[0], x, inputs["g_gamma"][lo:hi], level_mask=mask,
                          with_mags=False, nthreads=threads)


def siren_inputs(w, rank=0):
    """Seeded SIREN weights and upstream gradients for a Hermite workload."""
    from multiresolution_hash_grid_02_b300 import workloads as W
    rng = np.random.default_rng(w.seed + 2000 + rank)
    return W.siren_weights(rng, w.L * w.F), W.siren_upstream(rng, w.n_points, w.d)


def oracle_siren_step(oracle, w, res, tabs, inputs, sw, sup, lo, hi, mask, threads):
    """Oracle encoder + SIREN step on points [lo, hi): Hermite forward, SIREN
    forward and backward, Hermite backward of the SIREN's input gradients."""
    x = inputs["coords"][lo:hi]
    m, d, K = hi - lo, w.d, w.L * w.F
    enc = oracle.encode_fwd(w.d, w.F, res, w.log2_T, tabs, x, level_mask=mask, nthreads=threads, with_mags=False)
    feats = {"gamma": enc["gamma"].reshape(m, K), "dgamma": enc["dgamma"].reshape(m, d, K),
             "lap": enc["lap"].reshape(m, K)}
    from multiresolution_hash_grid_02_b300 import workloads as W
    oracle.siren_fwd(omega=W.SIREN_OMEGA, with_mags=False, **feats, **sw)
    g = oracle.siren_bwd(omega=W.SIREN_OMEGA, with_mags=False, **feats, **sw,
                         **{k: v[lo:hi] for k, v in sup.items()})
    oracle.encode_bwd(w.d, w.F, res, w.log2_T, x, g["g_gamma"].reshape(m, w.L, w.F),
                      g["g_dgamma"].reshape(m, d, w.L, w.F), g["g_lap"].reshape(m, w.L, w.F), level_mask=mask,
                      with_mags=False, nthreads=threads)


def cpu_baseline(w, inputs, mask, sample, hessian=False, siren=None):
    oracle, res, tabs = oracle_setup(w, inputs)
    threads = len(os.sched_getaffinity(0))
    sample = min(sample, w.n_points)

    def run(lo, hi):
        if siren:
            oracle_siren_step(oracle, w, res, tabs, inputs, siren[0], siren[1], lo, hi, mask, threads)
        else:
            oracle_step(oracle, w, res, tabs, inputs, lo, hi, mask, threads, hessian)
    run(0, min(256, sample))  # warm the code path
    t0 = time.perf_counter()
    run(0, sample)
    dt = time.perf_counter() - t0
    return {"value": sample / dt, "unit": "points/s", "cores": threads, "kind": "oracle",
            "sample": f"first {sample} of the {w.n_points} points, all {bin(mask).count('1')} active levels, "
                      f"fwd + bwd{' of encoder and SIREN' if siren else ''}, fp64, {dt:.1f} s"}


def run_reference(args):
    from multiresolution_hash_grid_02_b300 import workloads as W
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = W.WORKLOADS[args.config]
    mask = args.level_mask if args.level_mask is not None else (1 << w.L) - 1
    inputs = W.make(w)
    hessian = args.hessian and w.kind == "hermite"
    siren = siren_inputs(w) if (args.siren and w.kind == "hermite") else None
    if hessian:
        add_hessian_upstream(w, inputs)
    oracle, res, tabs = oracle_setup(w, inputs)
    threads = len(os.sched_getaffinity(0))
    per_step = min(max(256, args.cpu_sample // (32 if siren else 8)), w.n_points)
    times = []
    for i in range(args.warmup + args.steps):
        lo = (i * per_step) % max(1, w.n_points - per_step)
        t0 = time.perf_counter()
        if siren:
            oracle_siren_step(oracle, w, res, tabs, inputs, siren[0], siren[1], lo, lo + per_step, mask, threads)
        else:
            oracle_step(oracle, w, res, tabs, inputs, lo, lo + per_step, mask, threads, hessian)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    t = sum(times)
    value = per_step * len(times) / t
    line = {"impl": "reference", "metric": metric_of(w, hessian, siren is not None), "value": value, "unit": "points/s",
            "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded numpy)", "config": describe(w, mask, args.layout, hessian, siren is not None),
            "cpu_baseline": {"value": value, "unit": "points/s", "cores": threads, "kind": "oracle",
                             "sample": f"{per_step} points per step (of {w.n_points}), fwd + bwd"
                                       f"{' of encoder and SIREN' if siren else ''}, all active levels"},
            "e2e": {"value": value, "unit": "points/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# native (CUDA) arm
# ---------------------------------------------------------------------------

def kernel_patterns(w):
    """(row bytes, lanes per row) of the forward gather and the backward RED
    the kernels issue for this workload (packed layout)."""
    es = 2 if w.dtype == "f16" else 4
    slots = (1 << w.d) if w.kind == "hermite" else 1
    trow = slots * w.F * es
    grow = slots * w.F * 4
    # forward: lane pairs for 3D F = 2 rows (64 B fp32, 32 B fp16), lane quads for 4D F = 2 rows (128 B
    # fp32, 64 B fp16), one thread per row otherwise (Hermite rows with one vector load, d-linear F values)
    if w.kind == "hermite" and w.d == 3 and w.F == 2:
        g = (trow, 2)
    elif w.kind == "hermite" and w.d == 4 and w.F == 2:
        g = (trow, 4)
    else:
        g = (trow, 1)
    # backward: one 16-byte RED per lane and row for 32-128 B Hermite rows, one RED per row otherwise
    r = {128: (128, 8), 64: (64, 4), 32: (32, 2)}.get(grow, (grow, 1)) if w.kind == "hermite" else (grow, 1)
    return g, r


def replay_peaks(torch, hg, desc, n, coords, table, grad, gather_pat, red_pat, gather_bytes, red_bytes, stream):
    """Ceilings of the encoding kernels' own row streams: the memory-only
    replays hg_probe_replay_gather / hg_probe_replay_red run the launch's
    exact row addresses (same coordinates, levels, index function, packed
    rows) with the kernels' lane split and vector width and no arithmetic;
    ceiling = the kernel's algorithmic bytes / the replay's time (best of 3
    after one warm-up).  The RED replay writes into `grad`, which every step
    zeroes first."""
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def best(fn):
        t = float("inf")
        for i in range(4):
            ev[0].record(stream)
            fn()
            ev[1].record(stream)
            torch.cuda.synchronize()
            if i:
                t = min(t, ev[0].elapsed_time(ev[1]))
        return t

    (grow, glanes), (rrow, rlanes) = gather_pat, red_pat
    sink = torch.empty(n * glanes, device="cuda")
    tg = best(lambda: hg.hg_probe_replay_gather(desc, n, coords, table, table.stride(0) * table.element_size(),
                                                grow, glanes, sink, stream))
    tr = best(lambda: hg.hg_probe_replay_red(desc, n, coords, grad, grad.stride(0) * grad.element_size(), rrow,
                                             rlanes, stream))
    return gather_bytes / (tg * 1e-3) / 1e9, red_bytes / (tr * 1e-3) / 1e9, tg, tr


def probe_peaks(torch, hg, gather_pat, red_pat, log2_bytes=(25, 25)):
    """Measured ceilings for the kernels' own access patterns: random
    whole-row gathers and random 16-byte vector REDs on buffers of
    2^log2_bytes[0] and 2^log2_bytes[1] bytes (32 MiB: L2-resident; 1 GiB:
    HBM), rows split across lanes as the kernels split them; best of 5 after
    one warm-up launch."""
    if isinstance(log2_bytes, int):
        log2_bytes = (log2_bytes, log2_bytes)
    buf = torch.zeros(1 << (max(log2_bytes) - 2), dtype=torch.float32, device="cuda")
    n_threads = 148 * 2048 * 4
    sink = torch.empty(n_threads, device="cuda")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def best(fn, nbytes):
        b = 0.0
        for i in range(6):
            ev[0].record()
            fn(i)
            ev[1].record()
            torch.cuda.synchronize()
            if i:
                b = max(b, nbytes / (ev[0].elapsed_time(ev[1]) * 1e-3) / 1e9)
        return b

    grow, glanes = gather_pat
    rrow, rlanes = red_pat
    gl2 = log2_bytes[0] - {128: 7, 64: 6, 32: 5, 16: 4, 8: 3}[grow]
    rl2 = log2_bytes[1] - {128: 7, 64: 6, 32: 5, 16: 4, 8: 3}[rrow]
    per_g, per_r = 64, 64
    g = best(lambda i: hg.hg_probe_l2_gather(buf, gl2, grow, glanes, n_threads, per_g, i, sink),
             n_threads // glanes * per_g * grow)
    r = best(lambda i: hg.hg_probe_l2_red(buf, rl2, rrow, rlanes, n_threads, per_r, i),
             n_threads // rlanes * per_r * rrow)
    return g, r


def probe_pattern_table():
    """L2 random-row rates for every lanes-per-row split the probes support:
    the measurement behind splitting each (point, level) across lanes."""
    import torch
    from multiresolution_hash_grid_02_b300 import hg
    rows = {}
    for where, l2b in (("L2 (32 MiB)", 25), ("HBM (1 GiB)", 30)):
        for kind, pats in (("gather", ((32, 1), (32, 2), (64, 1), (64, 2), (64, 4))),
                           ("red", ((16, 1), (32, 1), (32, 2), (64, 1), (64, 2), (64, 4)))):
            for pat in pats:
                g, r = probe_peaks(torch, hg, pat if kind == "gather" else (64, 2), pat if kind == "red" else (64, 4),
                                   l2b)
                rows[f"{where} {kind} {pat[0]}-byte rows, {pat[1]} lane(s)/row"] = round(g if kind == "gather" else r, 1)
    return rows


def main():
    args = parse_args()
    if args.probe_patterns:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        print(json.dumps({"probe_patterns_gbs": probe_pattern_table(), "gpu": torch.cuda.get_device_name()}),
              flush=True)
        return
    if args.record_traffic:
        from multiresolution_hash_grid_02_b300 import workloads as W
        w = W.WORKLOADS[args.config]
        kern = "hermite_bwd" if args.record_traffic_kernel == "bwd" else "hermite_fwd"
        extra = (f" --config {args.config}" if args.config != 4 else "") + (" --hessian" if args.hessian else "") + \
            (f" --points {args.points}" if args.points else "")
        record_traffic(args.record_traffic, traffic_key(w, args.points, args.hessian),
                       "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum "
                       f"--clock-control none -k regex:{kern} -s 1 -c 1 python bench.py --steps 2 --warmup 1 "
                       "--no-e2e --no-cpu-baseline --no-all-configs" + extra)
        return
    if args.impl == "reference":
        run_reference(args)
        return
    if args.siren:
        run_siren(args)
        return
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from multiresolution_hash_grid_02_b300 import workloads as W

    w = W.WORKLOADS[args.config]
    if args.points:
        w = w.scaled(args.points)
    mask = args.level_mask if args.level_mask is not None else (1 << w.L) - 1
    hessian = args.hessian and w.kind == "hermite"
    line = measure_native(args, w, mask, hessian, world, rank, local, with_e2e=not args.no_e2e and rank == 0,
                          cpu_sample=None if (args.no_cpu_baseline or rank != 0 or world > 1) else args.cpu_sample)
    # the other workloads of the metric, each timed the same way (same steps and warm-up), reported inside
    # the headline line so that one run records them all; the headline's own keys keep their meaning
    if (rank == 0 and world == 1 and not args.no_all_configs and args.config == 4 and not hessian
            and args.points is None and args.level_mask is None):
        line["all_configs"] = all_configs(args)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# the workloads reported beside the headline (workload number, active levels or None = all)
OTHER_CONFIGS = ((1, None), (2, None), (3, None), (10, None), (5, 4), (5, 10), (5, 16))


def all_configs(args):
    """One compact record per other workload of the metric (the tiny 2D
    Hermite grid, the d-linear Instant-NGP grid, the PINN grid in stratum and
    in shuffled order, the large fp16 grid at L_active = 4, 10, 16): the
    device-timed step with its roofline and the oracle's CPU rate on a small
    sample.  A failure is recorded, not raised, so the headline still prints."""
    import torch
    from multiresolution_hash_grid_02_b300 import workloads as W
    out = []
    cache = {}
    for cfg, active in OTHER_CONFIGS:
        w = W.WORKLOADS[cfg]
        mask = (1 << w.L) - 1 if active is None else (1 << active) - 1
        try:
            if cache.get("cfg") != cfg:
                cache.clear()
                cache["cfg"], cache["inputs"] = cfg, W.make(w)
            ln = measure_native(args, w, mask, False, 1, 0, int(os.environ.get("LOCAL_RANK", "0")), with_e2e=False,
                                cpu_sample=None if args.no_cpu_baseline else min(w.n_points, 1 << 15),
                                inputs=cache["inputs"])
            out.append({"workload": w.name, "config_index": cfg, "active_levels": bin(mask).count("1"),
                        "value": ln["value"], "unit": ln["unit"], "ms_per_step": ln["ms_per_step"],
                        "ms_per_step_median": ln["ms_per_step_median"], "fwd_ms": ln["kernels"]["fwd"]["ms"],
                        "bwd_ms": ln["kernels"]["bwd"]["ms"], "fwd_frac": ln["kernels"]["fwd"]["frac"],
                        "bwd_frac": ln["kernels"]["bwd"]["frac"], "fwd_probe": ln["kernels"]["fwd"]["probe"],
                        "bwd_probe": ln["kernels"]["bwd"]["probe"],
                        "roofline": {k: ln["roofline"][k] for k in ("bound", "kernel", "achieved", "peak", "unit",
                                                                    "frac", "combined_frac", "traffic")},
                        "cpu_baseline": ln["cpu_baseline"], "clocks": ln["clocks"], "config": ln["config"]})
        except Exception as e:  # noqa: BLE001 -- recorded in the line
            out.append({"workload": w.name, "config_index": cfg, "active_levels": bin(mask).count("1"),
                        "error": f"{type(e).__name__}: {e}"})
        torch.cuda.empty_cache()
    return out


def measure_native(args, w, mask, hessian, world, rank, local, with_e2e, cpu_sample, inputs=None):
    """Time args.steps steps of one workload (after args.warmup untimed ones)
    and return the JSON record: whole-run throughput, per-kernel medians and
    rooflines, optional end-to-end leg and CPU baseline."""
    import torch
    import torch.distributed as dist
    from multiresolution_hash_grid_02_b300 import hg, workloads as W
    import multiresolution_hash_grid_02_b300 as M

    layout = M.HG_FEATURE_MAJOR if args.layout == "feature" else M.HG_POINT_MAJOR
    fm = layout == M.HG_FEATURE_MAJOR
    if inputs is None:
        inputs = W.make(w, seed=w.seed + rank)
    if hessian:
        add_hessian_upstream(w, inputs, rank)
    n, d, L, F = w.n_points, w.d, w.L, w.F
    P = d * (d + 1) // 2
    desc = M.GridDesc(d=d, L=L, F=F, n_min=w.n_min, n_max=w.n_max, log2_T=w.log2_T * (d + 1) if w.kind != "hermite"
                      else w.log2_T, level_mask=mask, dtype=M.HG_F16 if w.dtype == "f16" else M.HG_F32, layout=layout)

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    coords = dev(inputs["coords"])
    table = dev(inputs["table"])
    hermite = w.kind == "hermite"
    rbf = w.kind == "rbf"
    conv = (lambda a, ax: W.to_feature_major(a, ax)) if fm else (lambda a, ax: a)
    gg = dev(conv(inputs["g_gamma"], False))
    gd = dev(conv(inputs["g_dgamma"], True)) if (hermite or rbf) else None
    shape_g = (L, F, n) if fm else (n, L, F)
    shape_d = (d, L, F, n) if fm else (n, d, L, F)
    # second-order output and its upstream gradient: the Laplacian, or the full Hessian
    shape_s = ((P, L, F, n) if fm else (n, P, L, F)) if hessian else shape_g
    gl = (dev(conv(inputs["g_hess"], True)) if hessian else dev(conv(inputs["g_lap"], False))) if (hermite or rbf) \
        else None
    fd = w.kind == "linear_fd"
    shape_st = (2 * d, L, F, n) if fm else (n, 2 * d, L, F)          # INGP-FD stencil encodings
    gst = dev(conv(inputs["g_stencil"], True)) if fd else None
    stencil = torch.empty(shape_st, device="cuda") if fd else None
    gamma = torch.empty(shape_g, device="cuda")
    dgamma = torch.empty(shape_d, device="cuda") if (hermite or rbf) else None
    lap = torch.empty(shape_s, device="cuda") if (hermite or rbf) else None
    grad = torch.zeros(table.shape, dtype=torch.float32, device="cuda")
    if hermite:
        tviews, gviews = M.packed_views(table, d), M.packed_views(grad, d)
    else:
        tviews, gviews = M.linear_view(table), M.linear_view(grad)
    stream = torch.cuda.current_stream()

    def fwd():
        if hessian:
            hg.hg_encode_fwd_hessian(desc, n, coords, tviews, gamma, dgamma, lap, stream)
        elif hermite:
            hg.hg_encode_fwd(desc, n, coords, tviews, gamma, dgamma, lap, stream)
        elif fd:
            hg.hg_linear_fd_fwd(desc, n, coords, w.eps, tviews, gamma, None, None, stencil, stream)
        elif rbf:
            hg.hg_rbf_fwd(desc, n, coords, w.eps, w.rings, tviews, gamma, dgamma, lap, stream)
        else:
            hg.hg_linear_fwd(desc, n, coords, tviews, gamma, stream)

    def bwd():
        if hessian:
            hg.hg_encode_bwd_hessian(desc, n, coords, gg, gd, gl, gviews, stream)
        elif hermite:
            hg.hg_encode_bwd(desc, n, coords, gg, gd, gl, gviews, stream)
        elif fd:
            hg.hg_linear_fd_bwd(desc, n, coords, w.eps, gg, None, None, gst, gviews, stream)
        elif rbf:
            hg.hg_rbf_bwd(desc, n, coords, w.eps, w.rings, gg, gd, gl, gviews, stream)
        else:
            hg.hg_linear_bwd(desc, n, coords, gg, gviews, stream)

    launches_per_step = 2
    # per step: before the zeroing, before the forward, between, after the backward
    ev_f = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]

    def step(rec=None):
        if rec:
            rec[0].record(stream)
        grad.zero_()
        if rec:
            rec[1].record(stream)
        fwd()
        if rec:
            rec[2].record(stream)
        bwd()
        if rec:
            rec[3].record(stream)

    gather_pat, red_pat = kernel_patterns(w)
    gather_bytes, red_bytes = algorithmic_bytes(w, mask)
    if rbf:   # the replay probes replay 2^d-corner streams, not the RBF's ring box
        gather_peak = red_peak = 0.0
        t_replay_g = t_replay_r = float("nan")
    else:
        gather_peak, red_peak, t_replay_g, t_replay_r = replay_peaks(torch, hg, desc, n, coords, table, grad,
                                                                     gather_pat, red_pat, gather_bytes, red_bytes,
                                                                     stream)
    uniform_g, uniform_r = probe_peaks(torch, hg, gather_pat, red_pat)
    # the ceiling is the larger of the two measured rates: the replay of the exact stream, and the
    # contention-free uniform-random rate of the same row pattern, which kernels that sum
    # contributions on chip before the RED (run aggregation, privatised levels) can approach
    replay_g, replay_r = gather_peak, red_peak
    gather_peak, red_peak = max(replay_g, uniform_g), max(replay_r, uniform_r)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(ev_f[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), world, "cuda")
    # per-launch durations: the median over the timed steps of each launch's events
    t_fwd = statistics.median(e[1].elapsed_time(e[2]) for e in ev_f)
    t_bwd = statistics.median(e[2].elapsed_time(e[3]) for e in ev_f)
    t_step_med = statistics.median(e[0].elapsed_time(e[3]) for e in ev_f)

    total_points = n * world * args.steps
    value = total_points / (elapsed_ms * 1e-3)

    fwd_gbs = gather_bytes / (t_fwd * 1e-3) / 1e9
    bwd_gbs = red_bytes / (t_bwd * 1e-3) / 1e9
    t_bound = gather_bytes / (gather_peak * 1e9) + red_bytes / (red_peak * 1e9)
    combined = t_bound / ((t_fwd + t_bwd) * 1e-3)
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    hbm = None
    if os.path.exists(peaks_path):
        with open(peaks_path) as f:
            hbm = json.load(f).get("hbm_gbs")
    kernels = {
        "fwd": {"ms": t_fwd, "bound": "l2", "achieved": fwd_gbs, "peak": gather_peak, "unit": "GB/s",
                "frac": fwd_gbs / gather_peak, "algorithmic_bytes": gather_bytes,
                "probe": f"{gather_pat[0]}-byte rows, {gather_pat[1]} lane(s) per row; replay of this launch's "
                         f"row stream {t_replay_g:.3f} ms = {replay_g:.0f} GB/s, uniform random rows in 32 MiB "
                         f"{uniform_g:.0f} GB/s; peak = the larger",
                "what": "compulsory coefficient bytes gathered / median launch time vs the larger measured ceiling"},
        "bwd": {"ms": t_bwd, "bound": "l2", "achieved": bwd_gbs, "peak": red_peak, "unit": "GB/s",
                "frac": bwd_gbs / red_peak, "algorithmic_bytes": red_bytes,
                "probe": f"{red_pat[0]}-byte rows, {red_pat[1]} lane(s) per row; replay of this launch's "
                         f"row stream {t_replay_r:.3f} ms = {replay_r:.0f} GB/s, uniform random rows in 32 MiB "
                         f"{uniform_r:.0f} GB/s; peak = the larger",
                "what": "fp32 gradient RED payload bytes / median launch time vs the larger measured ceiling"},
    }
    if hbm:
        for key, ach in (("fwd", fwd_gbs), ("bwd", bwd_gbs)):
            kernels[key]["frac_of_hbm_peak"] = ach / hbm
    if rbf:
        # the RBF grids are small and L1/L2-resident: the kernels are bound on chip (arithmetic latency,
        # shared-memory atomics), so the roofline is FP32 arithmetic against the FMA peak at the sampled clock
        flops = rbf_flops(w, mask)
        fp32 = fp32_peak_tflops(torch, (clocks or {}).get("sm_mhz") or 2032.0)
        for key, t in (("fwd", t_fwd), ("bwd", t_bwd)):
            ach = flops / (t * 1e-3) / 1e12
            kernels[key].pop("frac_of_hbm_peak", None)
            kernels[key].update({"bound": "alu", "achieved": ach, "peak": fp32, "unit": "TFLOP/s",
                                 "frac": ach / fp32, "algorithmic_flops": flops,
                                 "probe": "FP32 FMA peak: SMs x 128 lanes x 2 flops x median sampled SM clock",
                                 "what": "separable-contraction flops / median launch time vs the FP32 FMA peak"})
        combined = (2 * flops / (fp32 * 1e12)) / ((t_fwd + t_bwd) * 1e-3)
    dom = "bwd" if t_bwd >= t_fwd else "fwd"
    k = kernels[dom]
    prefix = {"hermite": "hermite", "linear": "linear", "linear_fd": "linear_fd", "rbf": "rbf"}[w.kind]
    kname = {"fwd": prefix + "_fwd", "bwd": prefix + "_bwd"}[dom]
    traffic = recorded_traffic(traffic_key(w, args.points, hessian), kname)
    roofline = {"bound": k["bound"], "kernel": dom, "achieved": k["achieved"], "peak": k["peak"], "unit": k["unit"],
                "frac": k["frac"], "traffic": traffic,
                "peak_source": "measured live, the larger of: algorithmic bytes / time of hg_probe_replay_gather "
                               "or hg_probe_replay_red (the launch's own row addresses, lane split and vector "
                               "width, no arithmetic), and hg_probe_l2_gather / hg_probe_l2_red (uniform random "
                               "rows of the same size and split in an L2-resident 32 MiB buffer)",
                "combined_frac": combined, "hbm_peak_gbs": hbm,
                "frac_of_hbm_peak": k.get("frac_of_hbm_peak")}
    if rbf:
        roofline["peak_source"] = ("FP32 FMA peak (SMs x 128 lanes x 2 flops x the median SM clock sampled during the "
                                   "timed region); achieved = the separable contraction's flops / launch time")

    e2e = None
    if with_e2e:
        e2e = run_e2e(torch, hg, M, W, w, desc, inputs, tviews, gviews, conv, shape_g, shape_d, shape_s, hermite,
                      hessian, grad, stream, shape_st, steps=args.steps, warmup=max(2, args.warmup))
    cpu = None
    if cpu_sample:
        cpu = cpu_baseline(w, inputs, mask, cpu_sample, hessian)

    return {
        "metric": metric_of(w, hessian), "value": value, "unit": "points/s", "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "ms_per_step_median": t_step_med,
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded numpy: uniform coords, uniform coefficients, N(0,1) upstream gradients)",
        "config": describe(w, mask, args.layout, hessian),
        "roofline": roofline, "kernels": kernels,
        "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }


def run_e2e(torch, hg, M, W, w, desc, inputs, tviews, gviews, conv, shape_g, shape_d, shape_s, hermite, hessian,
            grad, stream, shape_st=None, steps=8, warmup=2):
    """The step through the C ABI with inputs starting in pinned host memory,
    pipelined over three streams as a streaming user would run it: the
    host-to-device copy of step i+1's coordinates and upstream gradients and
    the device-to-host read of step i-1's gamma / grad gamma / Laplacian
    overlap the encode of step i (two device buffer sets).  Every step's
    copies and kernels are inside the timed region.  With `hessian` the
    second-order output and upstream are the full Hessian's (shape_s)."""
    n = w.n_points

    def pinned(a):
        return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()

    h_in = [pinned(inputs["coords"]), pinned(conv(inputs["g_gamma"], False))]
    rbf = w.kind == "rbf"
    if hermite or rbf:
        second = conv(inputs["g_hess"], True) if hessian else conv(inputs["g_lap"], False)
        h_in += [pinned(conv(inputs["g_dgamma"], True)), pinned(second)]
    fd = w.kind == "linear_fd"
    if fd:
        h_in += [pinned(conv(inputs["g_stencil"], True))]
    out_shapes = [shape_g] + ([shape_d, shape_s] if (hermite or rbf) else []) + ([shape_st] if fd else [])
    d_in = [[torch.empty_like(t, device="cuda") for t in h_in] for _ in range(2)]
    d_out = [[torch.empty(sh, device="cuda") for sh in out_shapes] for _ in range(2)]
    h_out = [[torch.empty(sh).pin_memory() for sh in out_shapes] for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out[0])
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    s_comp = stream
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    started = [False, False]

    def step(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            if started[b]:
                s_in.wait_event(ev_comp[b])          # step i-2 has finished reading this input set
            for d, h in zip(d_in[b], h_in):
                d.copy_(h, non_blocking=True)
            ev_in[b].record(s_in)
        s_comp.wait_event(ev_in[b])
        if started[b]:
            s_comp.wait_event(ev_out[b])             # step i-2's outputs are on the host
        grad.zero_()
        c, gg = d_in[b][0], d_in[b][1]
        if hessian:
            hg.hg_encode_fwd_hessian(desc, n, c, tviews, d_out[b][0], d_out[b][1], d_out[b][2], s_comp)
            hg.hg_encode_bwd_hessian(desc, n, c, gg, d_in[b][2], d_in[b][3], gviews, s_comp)
        elif hermite:
            hg.hg_encode_fwd(desc, n, c, tviews, d_out[b][0], d_out[b][1], d_out[b][2], s_comp)
            hg.hg_encode_bwd(desc, n, c, gg, d_in[b][2], d_in[b][3], gviews, s_comp)
        elif rbf:
            hg.hg_rbf_fwd(desc, n, c, w.eps, w.rings, tviews, d_out[b][0], d_out[b][1], d_out[b][2], s_comp)
            hg.hg_rbf_bwd(desc, n, c, w.eps, w.rings, gg, d_in[b][2], d_in[b][3], gviews, s_comp)
        elif fd:
            hg.hg_linear_fd_fwd(desc, n, c, w.eps, tviews, d_out[b][0], None, None, d_out[b][1], s_comp)
            hg.hg_linear_fd_bwd(desc, n, c, w.eps, gg, None, None, d_in[b][2], gviews, s_comp)
        else:
            hg.hg_linear_fwd(desc, n, c, tviews, d_out[b][0], s_comp)
            hg.hg_linear_bwd(desc, n, c, gg, gviews, s_comp)
        ev_comp[b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[b])
            for h, d in zip(h_out[b], d_out[b]):
                h.copy_(d, non_blocking=True)
            ev_out[b].record(s_out)
        started[b] = True

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(warmup, warmup + steps):
        step(i)
    e.record(s_out)
    torch.cuda.synchronize()
    ms = a.elapsed_time(e) / steps
    return {"value": n / (ms * 1e-3), "unit": "points/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": ms, "steps": steps,
            "note": "pinned host buffers; coordinates and upstream gradients in, "
                    + ("gamma and the stencil encodings" if w.kind == "linear_fd" else
                       "gamma/grad gamma/" + ("Hessian" if hessian else "Laplacian")) + " out, "
                    "every step; copies of neighbouring steps overlap the encode (3 streams, 2 buffer sets); "
                    "gradient tables stay on the device"}


def run_siren(args):
    """The encoder + SIREN step (native arm): Hermite forward into the
    feature-major gamma, grad gamma and Laplacian; the SIREN forward (u, grad
    u, lap u); the SIREN backward from N(0,1) upstream gradients of those
    (input gradients and weight gradients); the Hermite backward of the input
    gradients.  Four launches of this library per step."""
    import torch
    import torch.distributed as dist
    from multiresolution_hash_grid_02_b300 import hg, workloads as W
    import multiresolution_hash_grid_02_b300 as M

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    w = W.WORKLOADS[args.config]
    if w.kind != "hermite":
        raise SystemExit("--siren needs a Hermite workload (it consumes gamma, grad gamma and lap gamma)")
    if args.points:
        w = w.scaled(args.points)
    mask = args.level_mask if args.level_mask is not None else (1 << w.L) - 1
    inputs = W.make(w, seed=w.seed + rank)
    sw, sup = siren_inputs(w, rank)
    n, d, L, F = w.n_points, w.d, w.L, w.F
    K, H, O = L * F, W.SIREN_H, W.SIREN_O
    desc = M.GridDesc(d=d, L=L, F=F, n_min=w.n_min, n_max=w.n_max, log2_T=w.log2_T, level_mask=mask,
                      dtype=M.HG_F16 if w.dtype == "f16" else M.HG_F32, layout=M.HG_FEATURE_MAJOR)
    sdesc = M.SirenDesc(d=d, K=K, H=H, O=O, omega=W.SIREN_OMEGA)

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    def fmaj(a):  # point-major [n][...] -> feature-major [...][n]
        return np.ascontiguousarray(np.moveaxis(a, 0, -1))

    coords, table = dev(inputs["coords"]), dev(inputs["table"])
    grad = torch.zeros(table.shape, dtype=torch.float32, device="cuda")
    tviews, gviews = M.packed_views(table, d), M.packed_views(grad, d)
    W1, b1, W2, b2 = (dev(sw[k]) for k in ("W1", "b1", "W2", "b2"))
    g_u, g_du, g_lapu = (dev(fmaj(sup[k])) for k in ("g_u", "g_du", "g_lapu"))
    gamma, dgamma, lap = (torch.empty(sh, device="cuda") for sh in ((L, F, n), (d, L, F, n), (L, F, n)))
    u, du, lapu = (torch.empty(sh, device="cuda") for sh in ((O, n), (d, O, n), (O, n)))
    gg, gd, gl = (torch.empty(sh, device="cuda") for sh in ((L, F, n), (d, L, F, n), (L, F, n)))
    gW1, gb1, gW2, gb2 = (torch.zeros(sh, device="cuda") for sh in ((H, K), (H,), (O, H), (O,)))
    stream = torch.cuda.current_stream()

    def step(rec=None):
        grad.zero_()
        for t in (gW1, gb1, gW2, gb2):
            t.zero_()
        if rec:
            rec[0].record(stream)
        hg.hg_encode_fwd(desc, n, coords, tviews, gamma, dgamma, lap, stream)
        if rec:
            rec[1].record(stream)
        hg.hg_siren_fwd(sdesc, n, gamma, dgamma, lap, W1, b1, W2, b2, u, du, lapu, stream)
        if rec:
            rec[2].record(stream)
        hg.hg_siren_bwd(sdesc, n, gamma, dgamma, lap, W1, b1, W2, g_u, g_du, g_lapu, gg, gd, gl, gW1, gb1, gW2,
                        gb2, stream)
        if rec:
            rec[3].record(stream)
        hg.hg_encode_bwd(desc, n, coords, gg, gd, gl, gviews, stream)
        if rec:
            rec[4].record(stream)

    gather_pat, red_pat = kernel_patterns(w)
    gather_bytes, red_bytes = algorithmic_bytes(w, mask)
    replay_g, replay_r, t_replay_g, t_replay_r = replay_peaks(torch, hg, desc, n, coords, table, grad, gather_pat,
                                                              red_pat, gather_bytes, red_bytes, stream)
    uniform_g, uniform_r = probe_peaks(torch, hg, gather_pat, red_pat)
    gather_peak, red_peak = max(replay_g, uniform_g), max(replay_r, uniform_r)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(ev[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), world, "cuda")
    names = ("encode_fwd", "siren_fwd", "siren_bwd", "encode_bwd")
    ms = {nm: statistics.median(e[i].elapsed_time(e[i + 1]) for e in ev) for i, nm in enumerate(names)}
    fp32 = fp32_peak_tflops(torch, (clocks or {}).get("sm_mhz") or 2032.0)
    fl = siren_flops(n, d, K, H)
    kernels = {
        "encode_fwd": {"ms": ms["encode_fwd"], "bound": "l2", "peak": gather_peak, "unit": "GB/s",
                       "achieved": gather_bytes / (ms["encode_fwd"] * 1e-3) / 1e9, "algorithmic_bytes": gather_bytes},
        "siren_fwd": {"ms": ms["siren_fwd"], "bound": "alu", "peak": fp32, "unit": "TFLOP/s",
                      "achieved": fl / (ms["siren_fwd"] * 1e-3) / 1e12, "algorithmic_flops": fl},
        "siren_bwd": {"ms": ms["siren_bwd"], "bound": "alu", "peak": fp32, "unit": "TFLOP/s",
                      "achieved": 3 * fl / (ms["siren_bwd"] * 1e-3) / 1e12, "algorithmic_flops": 3 * fl},
        "encode_bwd": {"ms": ms["encode_bwd"], "bound": "l2", "peak": red_peak, "unit": "GB/s",
                       "achieved": red_bytes / (ms["encode_bwd"] * 1e-3) / 1e9, "algorithmic_bytes": red_bytes},
    }
    for k in kernels.values():
        k["frac"] = k["achieved"] / k["peak"]
    dom = max(kernels, key=lambda nm: kernels[nm]["ms"])
    k = kernels[dom]
    roofline = {"bound": k["bound"], "kernel": dom, "achieved": k["achieved"], "peak": k["peak"], "unit": k["unit"],
                "frac": k["frac"], "traffic": recorded_traffic(traffic_key(w, args.points) + "+siren", dom),
                "peak_source": ("FP32 FMA peak (SMs x 128 lanes x 2 flops x the median SM clock sampled during the "
                                "timed region); achieved = the SIREN contractions' flops / launch time")
                if k["bound"] == "alu" else
                ("measured live, the larger of the replay of the launch's own row stream and the uniform-random "
                 "L2 rate of the same row pattern")}
    # the fused forward (encoding formed on chip and fed to the first layer) beside the unfused pair
    fused = None
    if w.d in (2, 3) and w.F == 2:
        fu, fdu, flu = (torch.empty(sh, device="cuda") for sh in ((O, n), (d, O, n), (O, n)))

        def fused_fwd():
            hg.hg_encode_siren_fwd(desc, n, coords, tviews, sdesc, W1, b1, W2, b2, fu, fdu, flu, stream)
        for _ in range(args.warmup):
            fused_fwd()
        fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for a, b in fev:
            a.record(stream)
            fused_fwd()
            b.record(stream)
        torch.cuda.synchronize()
        fms = statistics.median(a.elapsed_time(b) for a, b in fev)
        unf = ms["encode_fwd"] + ms["siren_fwd"]
        fused = {"ms": fms, "unfused_ms": unf, "speedup": unf / fms,
                 "achieved_tflops_first_layer": fl / (fms * 1e-3) / 1e12, "peak_fp32_tflops": fp32,
                 "frac_fp32_first_layer_only": fl / (fms * 1e-3) / 1e12 / fp32,
                 "hbm_bytes_saved_per_step": 2 * n * (d + 2) * K * 4,
                 "what": "hg_encode_siren_fwd (one launch: encode every level of a tile of points into shared "
                         "memory, then the SIREN forward) vs hg_encode_fwd + hg_siren_fwd (gamma, grad gamma, "
                         "lap gamma written to and read back from HBM); median of the same steps"}
    e2e = None
    if not args.no_e2e and rank == 0:
        e2e = run_e2e_siren(torch, hg, w, desc, sdesc, inputs, sup, tviews, gviews, grad, (W1, b1, W2, b2),
                            (gW1, gb1, gW2, gb2), stream, steps=args.steps, warmup=max(2, args.warmup))
    cpu = None
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        cpu = cpu_baseline(w, inputs, mask, min(args.cpu_sample, 1 << 17), siren=(sw, sup))
    if rank == 0:
        line = {
            "metric": METRIC_SIREN, "value": n * world * args.steps / (elapsed_ms * 1e-3), "unit": "points/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded numpy: uniform coords and coefficients, SIREN initialisation, N(0,1) "
                    "upstream gradients of u, grad u, lap u)",
            "config": describe(w, mask, "feature", siren=True),
            "roofline": roofline, "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": 4 * args.steps, "clocks": clocks, "fused_forward": fused,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_e2e_siren(torch, hg, w, desc, sdesc, inputs, sup, tviews, gviews, grad, weights, wgrads, stream, steps=8,
                  warmup=2):
    """The encoder + SIREN step through the C ABI from pinned host memory:
    every step copies in the coordinates and the upstream gradients of u,
    grad u and lap u, and copies out u, grad u and lap u; copies of
    neighbouring steps overlap the kernels (three streams, two buffer sets),
    as in the encoder's end-to-end leg."""
    n, d, L, F, O = w.n_points, w.d, w.L, w.F, sdesc.O

    def pinned(a):
        return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()

    h_in = [pinned(inputs["coords"])] + [pinned(np.moveaxis(sup[k], 0, -1)) for k in ("g_u", "g_du", "g_lapu")]
    out_shapes = [(O, n), (d, O, n), (O, n)]
    d_in = [[torch.empty_like(t, device="cuda") for t in h_in] for _ in range(2)]
    d_out = [[torch.empty(sh, device="cuda") for sh in out_shapes] for _ in range(2)]
    h_out = [[torch.empty(sh).pin_memory() for sh in out_shapes] for _ in range(2)]
    enc = [torch.empty(sh, device="cuda") for sh in ((L, F, n), (d, L, F, n), (L, F, n))]
    genc = [torch.empty(sh, device="cuda") for sh in ((L, F, n), (d, L, F, n), (L, F, n))]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out[0])
    s_in, s_out, s_comp = torch.cuda.Stream(), torch.cuda.Stream(), stream
    ev_in, ev_comp, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))
    started = [False, False]
    W1, b1, W2, b2 = weights

    def step(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            if started[b]:
                s_in.wait_event(ev_comp[b])
            for dd, h in zip(d_in[b], h_in):
                dd.copy_(h, non_blocking=True)
            ev_in[b].record(s_in)
        s_comp.wait_event(ev_in[b])
        if started[b]:
            s_comp.wait_event(ev_out[b])
        grad.zero_()
        for t in wgrads:
            t.zero_()
        c, gu, gdu, glu = d_in[b]
        hg.hg_encode_fwd(desc, n, c, tviews, enc[0], enc[1], enc[2], s_comp)
        hg.hg_siren_fwd(sdesc, n, enc[0], enc[1], enc[2], W1, b1, W2, b2, d_out[b][0], d_out[b][1], d_out[b][2],
                        s_comp)
        hg.hg_siren_bwd(sdesc, n, enc[0], enc[1], enc[2], W1, b1, W2, gu, gdu, glu, genc[0], genc[1], genc[2],
                        *wgrads, s_comp)
        hg.hg_encode_bwd(desc, n, c, genc[0], genc[1], genc[2], gviews, s_comp)
        ev_comp[b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[b])
            for h, dd in zip(h_out[b], d_out[b]):
                h.copy_(dd, non_blocking=True)
            ev_out[b].record(s_out)
        started[b] = True

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(warmup, warmup + steps):
        step(i)
    e.record(s_out)
    torch.cuda.synchronize()
    ms = a.elapsed_time(e) / steps
    return {"value": n / (ms * 1e-3), "unit": "points/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": ms, "steps": steps,
            "note": "pinned host buffers; coordinates and the upstream gradients of u, grad u, lap u in, u, grad u, "
                    "lap u out, every step; copies of neighbouring steps overlap the kernels (3 streams, 2 buffer "
                    "sets); the encoder outputs, gradient table and weight gradients stay on the device"}


if __name__ == "__main__":
    main()
