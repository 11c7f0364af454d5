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


def test_pool_leaves_at_least_four_timed_runs():
    assert bench.pool_size(32, 20) == 5            # the driver's short run: 4 runs
    assert bench.pool_size(32, 3200) == 32
    assert bench.pool_size(32, 3) == 1
    for steps in range(4, 200):
        assert -(-steps // bench.pool_size(32, steps)) >= 4


def test_code_digest_ignores_comments_only():
    src = 'int a = 1; // note\n/* block\n note */ const char* s = "//kept"; char c = \'/\';\n'
    assert bench.strip_comments(src) == 'int a = 1; const char* s = "//kept"; char c = \'/\';'
    assert bench.strip_comments("x = 1;   // one\n") == bench.strip_comments("x = 1;\n")
    assert bench.strip_comments("x = 1;") != bench.strip_comments("x = 2;")


def test_traffic_applies_only_to_its_workload(tmp_path, monkeypatch):
    import json
    import os
    os.makedirs(tmp_path / "profiles")
    digest = bench.source_digest()
    table = {"k_grad_norm_partial": {"dram_bytes_per_launch": 7, "source_digest": digest},
             "k_to_f32": {"dram_bytes_per_launch": 9, "source_digest": digest,
                          "workload": "andrea120m_fp16"},
             "k_grad_scale": {"dram_bytes_per_launch": 5, "source_digest": "0" * 16}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(table))
    real_root = bench.ROOT
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_digest", lambda read=None: digest)
    assert bench.traffic_from_profile("k_grad_norm_partial", "split", "andrea120m") == 7
    assert bench.traffic_from_profile("k_grad_norm_partial", "split", "andrea120m_fp16_inf") is None
    assert bench.traffic_from_profile("k_to_f32", "split", "andrea120m_fp16") == 9
    assert bench.traffic_from_profile("k_to_f32", "split", "andrea120m") is None
    assert bench.traffic_from_profile("k_grad_scale", "split", "andrea120m") is None  # stale
    assert real_root != str(tmp_path)
