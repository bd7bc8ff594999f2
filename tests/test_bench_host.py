"""bench.py's host-only legs: the one-thread oracle sample runs in a child process with the
BLAS/OpenMP thread counts set to 1 and reports that count (no GPU involved)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_oracle_sample_one_thread():
    sys.path.insert(0, ROOT)
    import bench
    r = bench.oracle_one_thread("tiny_mixed_s40", 0.2)
    assert "unavailable" not in r, r
    assert r["cores"] == 1
    assert r["value"] > 0 and r["seconds"] > 0
    assert "tiny_mixed_s40" in r["sample"]


def test_oracle_sample_flag_prints_json():
    env = dict(os.environ, OPENBLAS_NUM_THREADS="2", OMP_NUM_THREADS="2", CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--oracle-sample", "0.1",
                          "--workload", "tiny_mixed_s40"], env=env, capture_output=True,
                         text=True, timeout=300, check=True).stdout
    d = json.loads(out.strip().splitlines()[-1])
    assert d["flops"] > 0 and d["seconds"] > 0
    # threadpoolctl (when installed) reports the BLAS pool, else the variables are read
    assert 1 <= d["threads"] <= 2
