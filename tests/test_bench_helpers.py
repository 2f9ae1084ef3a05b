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
    # None once the kernel code differs from the summary's (re-profile then)
    row = bench.recorded_traffic("heterogeneous decode B=64 V=128256 bf16")
    fused = bench.recorded_traffic("fused LM head + draw B=64 d=4096 V=128256 bf16", "ss_fused_kernel")
    assert row is None or 16_000_000 < row < 18_000_000
    assert fused is None or 1_050_000_000 < fused < 1_060_000_000
    assert bench.recorded_traffic("some other workload") is None
