"""The benchmark's JSON contract, checked on the CPU: the reference arm (the
CPU oracle timed on a sample of the workload) prints one JSON line with the
required keys, and the GEMM traffic figure is withheld once the kernel
source no longer matches the capture it came from."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

REQUIRED = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
            "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"}


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "3"], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert REQUIRED <= set(d), REQUIRED - set(d)
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"] and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["config"]["workload"].startswith("tiny")
    # the reference arm's config is the one this build's line carries
    sys.path.insert(0, ROOT)
    import bench
    import fp8_workloads as wl
    assert d["config"] == bench.workload_config(wl.WORKLOADS["tiny"], 1)
    assert d["config"]["parallelism"] == "dp1 replicas"


def test_headline_defaults_to_the_largest_layer():
    """With no flags the headline is the 70B-shaped layer (M 8192, K 8192,
    N 28672), the largest single-GPU configuration."""
    sys.path.insert(0, ROOT)
    import bench
    old = sys.argv
    try:
        sys.argv = ["bench.py"]
        args = bench.parse_args()
    finally:
        sys.argv = old
    assert args.workload == "mlp70b" and args.gpus == 1
    import fp8_workloads as wl
    w = wl.WORKLOADS[args.workload]
    assert (w.M, w.K, w.N) == (8192, 8192, 28672) and w.margin == 1
    assert abs(bench.clock_peak(152 * 16384 * 1e6 / 1e12, 2070.0) - 5155.06176) < 1e-6
    assert bench.clock_peak(1.0, None) is None


def test_traffic_figure_follows_the_kernel_source(tmp_path, monkeypatch):
    """bench.gemm_traffic reports a capture's DRAM bytes only while the sha256
    it records matches the current gemm.cu."""
    import hashlib
    sys.path.insert(0, ROOT)
    import bench
    gemm_src = open(os.path.join(ROOT, "fp8_mixed_precision_amax_gb300", "csrc", "gemm.cu"),
                    "rb").read()
    prof = tmp_path / "profiles"
    prof.mkdir()
    pkg = tmp_path / "fp8_mixed_precision_amax_gb300" / "csrc"
    pkg.mkdir(parents=True)
    (pkg / "gemm.cu").write_bytes(gemm_src)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = {"kernel": "gemm_tn_kernel", "workload": "mlp7b", "bytes_per_launch_mean": 123.0,
           "gemm_cu_sha256": hashlib.sha256(gemm_src).hexdigest()}
    (prof / "gemm_tn_kernel.mlp7b.traffic.json").write_text(json.dumps(rec))
    assert bench.gemm_traffic("mlp7b") == 123.0
    # a capture of another source is not reported
    rec["gemm_cu_sha256"] = "0" * 64
    (prof / "gemm_tn_kernel.mlp7b.traffic.json").write_text(json.dumps(rec))
    assert bench.gemm_traffic("mlp7b") is None
    # nor is a workload without a capture
    assert bench.gemm_traffic("drift") is None


def test_range_counts_on_known_values():
    """The drift report's saturation / underflow counts, on values whose fate
    under E4M3 at scale 1 is fixed by the format (largest finite 448, smallest
    subnormal 2^-9, ties to even): 450, 512, -9984 and inf are clipped; 1e-5,
    -1e-6 and 2^-10 (exactly half the smallest subnormal, a tie that goes to
    the even code 0) become zero; 448, 2^-9, zeros and NaN are neither.  The
    oracle's cast of the same values must agree with that classification."""
    import numpy as np
    import torch
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import bench
    import oracle as o
    vals = [0.0, -0.0, 448.0, 450.0, 512.0, -9984.0, 1e-5, -1e-6, 2.0 ** -10, 2.0 ** -9,
            float("inf"), float("nan"), 1.0, -3.0]
    x = torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    codes, _ = o.quantize(bits[None, :], np.float32(1.0), o.E4M3)
    codes = codes.reshape(-1)
    sat, under = bench.range_counts(x, torch.from_numpy(codes.copy()), torch.ones(1), 448.0)
    assert (sat, under) == (4, 3)
    assert [int(c) & 0x7F for c in codes[[3, 4, 5, 10]]] == [0x7E] * 4
    assert [int(c) & 0x7F for c in codes[[6, 7, 8]]] == [0] * 3
    assert int(codes[9]) == 0x01 and int(codes[2]) == 0x7E


def test_range_counts_agree_with_the_oracle_cast():
    """On a seeded tensor with a scale that clips its tail and flushes its
    smallest values: every element counted as saturated is cast by the oracle
    to the largest-magnitude code, and the underflow count is the number of
    non-zero inputs the oracle casts to +-0."""
    import numpy as np
    import torch
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import bench
    import oracle as o
    g = torch.Generator().manual_seed(11)
    x = (torch.randn(64, 256, generator=g) * torch.logspace(-10, 1, 256)).to(torch.bfloat16)
    for fmt, fmax, s in ((o.E4M3, 448.0, 300.0), (o.E5M2, 57344.0, 1.0e4)):
        bits = x.view(torch.int16).numpy().view(np.uint16)
        codes, _ = o.quantize(bits, np.float32(s), fmt)
        sat, under = bench.range_counts(x, torch.from_numpy(codes.copy()),
                                        torch.tensor([s], dtype=torch.float32), fmax)
        top = 0x7E if fmt == o.E4M3 else 0x7B
        xd = o.bf16_to_f32(bits).astype(np.float64)
        exact = np.abs(xd * np.float64(np.float32(s)))
        assert sat > 0 and under > 0
        assert np.all((codes[exact > fmax] & 0x7F) == top)
        assert under == int(np.count_nonzero((xd != 0) & (o.fp8_decode_table(fmt)[codes] == 0)))


def test_clock_summary_from_nvidia_smi_lines():
    """The clocks object: median SM clock over samples under load (above half
    the maximum), the lowest of those, the peak power and every throttle
    reason seen Active in any sample; unparsable lines are skipped."""
    sys.path.insert(0, ROOT)
    import bench
    lines = ["2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active\n",
             "1605, 2070, 1391.0, 0x4, Not Active, Not Active, Not Active, Active\n",
             "1800, 2070, [N/A], 0x4, Not Active, Not Active, Not Active, Active\n",
             "345, 2070, 120.0, 0x0, Not Active, Not Active, Not Active, Not Active\n",
             "garbage\n", "N/A, N/A, N/A, N/A, N/A, N/A, N/A, N/A\n"]
    c = bench.ClockSampler.summarize(lines)
    assert c["samples"] == 4 and c["sm_max_mhz"] == 2070.0
    assert c["sm_mhz"] == 1800.0 and c["sm_min_mhz"] == 1605.0
    assert c["power_w_max"] == 1391.0
    assert c["reasons"] == ["sw_power_cap"]
    assert bench.ClockSampler.summarize([])["reasons"] == ["no samples"]


def test_reference_arm_under_torchrun_two_ranks():
    """With N = 2 ranks (gloo on the CPU), rank 0 alone times the oracle and
    prints one line, the other rank exits 0, and the oracle uses every core
    of rank 0's affinity mask although torchrun sets OMP_NUM_THREADS=1."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1", "--master-port",
                        str(port), "bench.py", "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "3", "--gpus", "2"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["cores"] == d["cpu_baseline"]["affinity_cores"] == \
        len(os.sched_getaffinity(0))
