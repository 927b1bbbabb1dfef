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


def test_traffic_figure_follows_the_kernel_source(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    assert bench.gemm_traffic("mlp7b") is not None      # the committed capture matches
    # a capture of another source is not reported
    prof = tmp_path / "profiles"
    prof.mkdir()
    src = json.load(open(os.path.join(ROOT, "profiles", "gemm_tn_kernel.mlp7b.traffic.json")))
    src["gemm_cu_sha256"] = "0" * 64
    (prof / "gemm_tn_kernel.mlp7b.traffic.json").write_text(json.dumps(src))
    pkg = tmp_path / "fp8_mixed_precision_amax_gb300" / "csrc"
    pkg.mkdir(parents=True)
    (pkg / "gemm.cu").write_bytes(open(os.path.join(ROOT, "fp8_mixed_precision_amax_gb300", "csrc",
                                                     "gemm.cu"), "rb").read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.gemm_traffic("mlp7b") is None
