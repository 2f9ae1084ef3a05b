"""Host-side helpers of the benchmark: the source hash that keys the recorded
ncu traffic ignores comments but not code, and the recorded traffic is read
only for its own workload."""
import bench


def test_code_only_hash_ignores_comments_not_code():
    a = "int f(int x) {\n  // twice\n  return 2 * x; /* doubled */\n}\n"
    b = "int f(int x) {\n  return 2 * x;\n}\n"
    c = "int f(int x) {\n  return 3 * x;\n}\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(b) != bench._code_only(c)
    assert "/*" not in bench._code_only("/* a\n multi-line\n comment */ int y;")


def test_recorded_traffic_is_read_for_its_workload_only():
    # None once the kernel code differs from the recorded entry's (re-profile then)
    row = bench.recorded_traffic("heterogeneous decode B=64 V=128256 bf16")
    fused = bench.recorded_traffic("fused LM head + draw B=64 d=4096 V=128256 bf16", "ss_fused_kernel")
    assert row is None or 16_000_000 < row < 18_000_000
    assert fused is None or 1_050_000_000 < fused < 1_060_000_000
    assert bench.recorded_traffic("some other workload") is None


def test_recorded_traffic_needs_the_current_source(tmp_path, monkeypatch):
    import json
    path = tmp_path / "traffic.json"
    entry = {"kernel": "ss_hist_kernel", "kernel_sha256": bench.kernel_source_hash("ss_hist_kernel"),
             "workload": "w", "traffic_bytes_per_launch": 123}
    path.write_text(json.dumps({"entries": [entry]}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(path))
    assert bench.recorded_traffic("w") == 123
    assert bench.recorded_traffic("w", "ss_fused_kernel") is None
    path.write_text(json.dumps({"entries": [dict(entry, kernel_sha256="0" * 16)]}))
    assert bench.recorded_traffic("w") is None


def test_launches_per_call():
    assert bench.launches_per_call({"dtype": "bf16", "kind": "sample", "num_rows": 64}, 4) == 1
    assert bench.launches_per_call({"dtype": "f32", "kind": "sample", "num_rows": 64}, 4) == 2
    assert bench.launches_per_call({"dtype": "f32", "kind": "sample", "num_rows": 4}, 1) == 1
