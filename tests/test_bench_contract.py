"""The benchmark's reference arm (the oracle on the host, no GPU) prints one
JSON line with the keys the contract asks for."""
import json
import os
import subprocess
import sys

from conftest import ROOT


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 2
    assert d["config"]["workload"].startswith("c3")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_traffic_record_follows_the_kernel_sources(tmp_path, monkeypatch):
    """The bench line's DRAM traffic comes from a capture record only while
    the kernel's sources are the ones it was taken on: a changed source byte,
    or another workload size, gives null."""
    import hashlib
    import shutil
    sys.path.insert(0, ROOT)
    import bench
    srcs = ["parity_binade_chunked_gb300/csrc/seqsum_kernel.cu", "parity_binade_chunked_gb300/csrc/binade_math.cuh",
            "parity_binade_chunked_gb300/csrc/seqsum_internal.cuh"]
    h = hashlib.sha256()
    for src in srcs:
        os.makedirs(os.path.dirname(tmp_path / src), exist_ok=True)
        shutil.copy(os.path.join(ROOT, src), tmp_path / src)
        h.update((tmp_path / src).read_bytes())
    os.makedirs(tmp_path / "profiles")
    rec = {"kernel_sources": srcs, "kernel_sources_sha256": h.hexdigest(),
           "dram_bytes_read_per_launch": 1000, "dram_bytes_write_per_launch": 24}
    (tmp_path / "profiles" / "seqsum_kernel_c3_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic("c3", 1) == 1024
    assert bench.measured_traffic("c3", 2) is None
    assert bench.measured_traffic("c5", 1) is None
    with open(tmp_path / srcs[1], "ab") as f:
        f.write(b"\n")
    assert bench.measured_traffic("c3", 1) is None
