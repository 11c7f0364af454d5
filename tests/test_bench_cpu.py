"""Host-side pieces of bench.py that need no GPU."""
import bench
import oracle
from workloads import WORKLOADS


def test_oracle_all_cores_runs_one_replica_per_core():
    oracle.build()
    r = bench.oracle_all_cores(WORKLOADS["tiny"], 0.2)
    assert "error" not in r, r
    assert r["cores"] >= 1 and r["value"] > 0 and r["kind"] == "oracle"


def test_algorithmic_bytes():
    assert bench.algorithmic_bytes(10, 4, "write") == 120
    assert bench.algorithmic_bytes(10, 2, "read") == 20
