"""Host-side logic of bench.py (no GPU): the multi-rank timing reduction over
world_size-2 gloo ranks, rank gating of the reference arm, the algorithmic
byte counts behind the roofline, and the recorded-traffic bookkeeping."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # each rank reports a different elapsed time; all must agree on the slowest
        q.put((rank, bench.max_over_ranks(10.0 + 7.5 * rank, world, "cpu")))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 17.5), (1, 17.5)]


def test_max_over_ranks_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert out.returncode == 0
    assert out.stdout.strip() == ""


def test_algorithmic_bytes_and_patterns():
    sys.path.insert(0, ROOT)
    import bench
    from multiresolution_hash_grid_02_b300 import workloads as W
    w = W.WORKLOADS[4]
    gather, red = bench.algorithmic_bytes(w, (1 << 16) - 1)
    # 2^21 points x 16 levels x 8 corners x (8 slots x 2 features x 4 bytes)
    assert gather == red == (1 << 21) * 16 * 8 * 64
    assert bench.algorithmic_bytes(w, 0b1111)[0] == gather // 4
    w5 = W.WORKLOADS[5]
    g5, r5 = bench.algorithmic_bytes(w5, (1 << 16) - 1)
    assert g5 == (1 << 23) * 16 * 8 * 32 and r5 == 2 * g5       # fp16 rows, fp32 gradients
    assert bench.kernel_patterns(w) == ((64, 2), (64, 4))
    assert bench.kernel_patterns(w5) == ((32, 2), (64, 4))
    w6 = W.WORKLOADS[6]
    # 4D: 2^20 points x 16 levels x 16 corners x (16 slots x 2 features x 4 bytes)
    assert bench.algorithmic_bytes(w6, (1 << 16) - 1) == ((1 << 20) * 16 * 16 * 128,) * 2
    assert bench.kernel_patterns(w6) == ((128, 4), (128, 8))
    w2 = W.WORKLOADS[2]
    assert bench.algorithmic_bytes(w2, (1 << 16) - 1) == ((1 << 20) * 16 * 4 * 8,) * 2
    assert bench.kernel_patterns(w2) == ((8, 1), (8, 1))          # d-linear: one float2 load / red.v2 per corner
    assert bench.kernel_patterns(W.WORKLOADS[3]) == ((32, 1), (32, 2))
    w7 = W.WORKLOADS[7]                                          # INGP-FD: the centre cell's 8-byte rows
    assert bench.algorithmic_bytes(w7, (1 << 16) - 1) == ((1 << 21) * 16 * 8 * 8,) * 2
    assert bench.kernel_patterns(w7) == ((8, 1), (8, 1))
    assert "INGP-FD" in bench.metric_of(w7) and bench.metric_of(w) != bench.metric_of(w7)
    # RBF: the ring box of taps; the separable contraction's flops (3D, 6 taps/axis: 6 (6 * 23 + 6) FMAs)
    w9 = W.WORKLOADS[9]
    assert bench.algorithmic_bytes(w9, 0b1111) == ((1 << 21) * 4 * 216 * 2 * 4,) * 2
    assert bench.rbf_flops(w9, 0b1111) == 2 * 864 * 2 * (1 << 21) * 4
    assert bench.rbf_flops(W.WORKLOADS[8], 0b1111) == 2 * 6 * 23 * 2 * (1 << 20) * 4
    assert "RBF" in bench.metric_of(w9)


def bench_workload(cfg):
    from multiresolution_hash_grid_02_b300 import workloads as W
    return W.WORKLOADS[cfg]


SAMPLE_NCU_LOG = """==PROF== Connected to process 1 (/usr/bin/python3.12)
==PROF== Profiling "hermite_fwd_pair3_kernel": 0%....50%....100% - 1 pass
{"metric": "ignored"}
  void unnamed>::hermite_fwd_pair3_kernel<float>(FwdParams) (16384, 16, 1)x(256, 1, 1), Context 1, Stream 7, Device 0, CC 10.3
    Section: Command line profiler metrics
    ---------------------------- ----------- ------------
    Metric Name                  Metric Unit Metric Value
    ---------------------------- ----------- ------------
    dram__bytes_read.sum              Mbyte       608.47
    dram__bytes_write.sum             Gbyte         1.31
    gpu__time_duration.sum               ms         2.37
  void unnamed>::hermite_bwd_split_kernel<3, 2, 4>(BwdParams) (32768, 16, 1)x(256, 1, 1), Context 1, Stream 7, Device 0, CC 10.3
    dram__bytes_read.sum              Gbyte         2.05
    dram__bytes_write.sum             Mbyte       287.08
"""


def test_ncu_log_parser_and_traffic_staleness(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    log = tmp_path / "ncu.log"
    log.write_text(SAMPLE_NCU_LOG)
    k = bench.parse_ncu_dram_log(str(log))
    assert set(k) == {"hermite_fwd_pair3_kernel<float>", "hermite_bwd_split_kernel<3, 2, 4>"}
    assert abs(k["hermite_fwd_pair3_kernel<float>"]["bytes_per_launch"] - (608.47e6 + 1.31e9)) < 1
    assert abs(k["hermite_bwd_split_kernel<3, 2, 4>"]["bytes_per_launch"] - (2.05e9 + 287.08e6)) < 1
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "traffic.json"))
    bench.record_traffic(str(log), "3d_hermite", "cmd")
    assert bench.recorded_traffic("3d_hermite", "hermite_bwd") == pytest.approx(2.05e9 + 287.08e6)
    assert bench.recorded_traffic("2d_hermite_pinn", "hermite_bwd") is None
    # a second configuration is kept beside the first
    bench.record_traffic(str(log), "3d_hermite+hessian", "cmd2")
    assert bench.recorded_traffic("3d_hermite", "hermite_fwd") == pytest.approx(608.47e6 + 1.31e9)
    assert bench.recorded_traffic("3d_hermite+hessian", "hermite_bwd") == pytest.approx(2.05e9 + 287.08e6)
    data = json.loads((tmp_path / "traffic.json").read_text())
    data["source_sha256"] = "0" * 64          # the kernels changed since the capture
    (tmp_path / "traffic.json").write_text(json.dumps(data))
    assert bench.recorded_traffic("3d_hermite", "hermite_bwd") is None
    assert bench.traffic_key(bench_workload(4), None, True) == "3d_hermite+hessian"


def test_traffic_hash_covers_the_hermite_sources_only(tmp_path, monkeypatch):
    """The recorded DRAM traffic stays valid across edits of kernels whose
    traffic is not recorded (the other encodings, the SIREN, the probes) and
    is invalidated by an edit of the Hermite kernels or their shared headers."""
    sys.path.insert(0, ROOT)
    import bench
    csrc = tmp_path / "multiresolution_hash_grid_02_b300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "include").mkdir()
    names = ["hermite_fwd.cu", "hermite_bwd.cu", "hg_device.cuh", "hg_params.h", "hg_api.cu"] + \
        list(bench.UNRECORDED_SOURCES)
    for nm in names:
        (csrc if nm != "hg_probe.h" else tmp_path / "include").joinpath(nm).write_text(nm)
    (tmp_path / "include" / "hg.h").write_text("hg.h")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    for nm in bench.UNRECORDED_SOURCES:
        f = (csrc if nm != "hg_probe.h" else tmp_path / "include") / nm
        f.write_text(nm + " edited")
        assert bench.kernel_source_hash() == h0, nm
    for f in (csrc / "hermite_fwd.cu", csrc / "hg_params.h", tmp_path / "include" / "hg.h"):
        old = f.read_text()
        f.write_text(old + " edited")
        assert bench.kernel_source_hash() != h0, f.name
        f.write_text(old)
    assert bench.kernel_source_hash() == h0


def test_reference_arm_fd_line():
    """The reference arm runs the INGP-FD workload's oracle step."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "7",
                          "--steps", "1", "--warmup", "0", "--cpu-sample", "4096"],
                         env=dict(os.environ, RANK="0", WORLD_SIZE="1"), capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert "INGP-FD" in line["metric"] and line["config"]["fd_eps"] == 2.0 ** -10 and line["value"] > 0


def test_reference_arm_hessian_line():
    """The reference arm (the oracle) runs the full-Hessian step on the tiny
    2D workload and labels its line accordingly."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "1",
                          "--hessian", "--steps", "1", "--warmup", "0", "--cpu-sample", "2048"],
                         env=dict(os.environ, RANK="0", WORLD_SIZE="1"), capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and "Hessian" in line["metric"]
    assert line["config"]["second_order"] == "full Hessian" and line["value"] > 0


def test_reference_arm_siren_line():
    """The reference arm runs the encoder + SIREN oracle step (workload 1: K = L F = 8)."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "1",
                          "--siren", "--steps", "1", "--warmup", "0", "--cpu-sample", "8192"],
                         env=dict(os.environ, RANK="0", WORLD_SIZE="1"), capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and "SIREN" in line["metric"] and line["value"] > 0
    assert line["config"]["siren_K"] == 8 and line["config"]["siren_omega"] == 30.0


def test_siren_flops():
    """The SIREN forward's algorithmic flops: its first layer, 2 (d + 2) K H per point."""
    import bench
    assert bench.siren_flops(1, 3, 32, 64) == 2 * 5 * 32 * 64
    assert bench.siren_flops(1 << 21, 2, 32, 64) == (1 << 21) * 2 * 4 * 32 * 64
