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


def test_decode_grid_count_follows_the_tail_rule():
    # pairs fill whole waves of the SMs; a last wave at most half full becomes a second
    # grid of key-split tiles (the launch rule of the decode call)
    sys.path.insert(0, ROOT)
    import bench
    assert bench.decode_grids(32, 4096, 1, 152) == 2       # 512 pairs: 56 left over
    assert bench.decode_grids(32, 16384, 2, 152) == 1      # 4096 pairs: 144 > 76 left over
    assert bench.decode_grids(3, 200, 4, 152) == 1         # 12 pairs: all key-split, one grid
    assert bench.decode_grids(8, 1024, 19, 152) == 1       # 608 pairs: 4 whole waves
    assert bench.decode_grids(8, 1000, 5, 152) == 2        # 160 pairs: 8 left over
    assert bench.decode_grids(1, 0, 1, 152) == 0           # nothing to launch
    # with a workspace: the balanced tail's pieces and merge behind the pair grid when a
    # range (plus 16 key tiles of overhead) is shorter than the tail's cost otherwise
    assert bench.decode_grids(32, 4096, 1, 152, 8384) == 3  # 56 pairs of 98 key tiles: 36 + 16 < 58.8
    assert bench.decode_grids(32, 4096, 1, 152, 256) == 2   # T2I, 34 key tiles: 12.5 + 16 > 20.4
    assert bench.decode_grids(4, 1000, 1, 152, 6000) == 2   # 16 pairs, all in the tail
    assert bench.decode_grids(4, 1000, 1, 152, 1100) == 1   # 17 key tiles per pair: key-split
    assert bench.decode_grids(32, 16384, 2, 152, 16968) == 1  # 144 pairs of 261: 247 + 16 > 261


def test_prefill_grid_count_follows_the_split_rule():
    # the pair grid, plus a key-split grid when at most four waves of pair CTAs, past
    # two whole waves, end in a partly filled one (the launch rule of the prefill call)
    sys.path.insert(0, ROOT)
    import bench
    assert bench.prefill_grids(32, 12480, 1, 152) == 1     # 8 x 49 x 4 = 1568 CTAs: 10 waves
    assert bench.prefill_grids(32, 4352, 1, 152) == 2      # 8 x 17 x 4 = 544: 88 left over
    assert bench.prefill_grids(16, 4096, 2, 152) == 2      # 8 x 16 x 4 = 512: 56 left over
    assert bench.prefill_grids(32, 2048, 1, 152) == 1      # 8 x 8 x 4 = 256: under two waves
    assert bench.prefill_grids(8, 9728, 1, 152) == 1       # 4 x 38 x 2 = 304: whole waves
    assert bench.prefill_grids(3, 40, 1, 152) == 1         # one pair per head


def test_reference_arm_line():
    # the reference arm times the oracle on the host and prints the contract's JSON line
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0", "--workload", "tiny_mixed_s40"],
                         env=env, capture_output=True, text=True, timeout=300, check=True).stdout
    d = json.loads(out.strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["higher_is_better"] is True
    assert d["unit"] == "TFLOP/s" and d["value"] > 0 and d["dtype"] == "f64"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"] == d["e2e"]["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "tiny_mixed_s40"


def test_clock_sampler_summary_and_bins():
    # nvidia-smi lines (index, sm, max, power, active, hw, hw_thermal, sw_thermal, sw_power)
    sys.path.insert(0, ROOT)
    import bench
    c = bench.ClockSampler(0)
    c.lines = ["0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
               "0, 1950, 2070, 1400.2, 0x4, Not Active, Not Active, Not Active, Active",
               "0, 1440, 2070, 1405.0, 0x4, Not Active, Not Active, Not Active, Active",
               "garbage"]
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 1950 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
    assert c.bins(60) == {"1440-1500": 1, "1920-1980": 1, "2040-2100": 1}
