"""bench.py's reference arm (the oracle on the host cores) prints one JSON line with the
keys of the bench contract, on the same metric, unit and workload as the GPU arm."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    sys.path.insert(0, ROOT)
    import bench
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == bench.WORKLOAD
    assert d["steps"] == 2 and d["warmup"] >= 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["vs_baseline"] is None
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_oracle_rows_cut_over_threads_change_no_bit(orc):
    """The all-core CPU baseline cuts the oracle's GEMV rows over host threads; every
    row is the same oracle computation, so the result equals one call bit for bit."""
    import concurrent.futures as cf
    import numpy as np
    g = np.random.default_rng(0)
    M, K, parts = 1001, 512, 7
    Wq = g.integers(-127, 128, size=(M, K)).astype(np.int8)
    Wd = g.integers(0x0c00, 0x1800, size=(M, K // 32)).astype(np.uint16)
    xq = g.integers(-127, 128, size=K).astype(np.int8)
    xd = g.integers(0x2000, 0x2c00, size=K // 32).astype(np.uint16)
    cuts = [M * j // parts for j in range(parts + 1)]
    with cf.ThreadPoolExecutor(max_workers=parts) as pool:
        y = np.concatenate(list(pool.map(lambda j: orc.gemv_q8_0(Wq[cuts[j]:cuts[j + 1]], Wd[cuts[j]:cuts[j + 1]],
                                                                 xq, xd), range(parts))))
    assert (y.view(np.uint64) == orc.gemv_q8_0(Wq, Wd, xq, xd).view(np.uint64)).all()
