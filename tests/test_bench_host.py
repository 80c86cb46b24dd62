"""Host-side pieces of bench.py that need no GPU: the kernel-source hash that decides
whether a recorded ncu traffic figure still describes the kernel, and the recorded
traffic lookup itself."""
import bench


def test_code_only_ignores_comments_and_blank_lines():
    code = "int a = 1;\nint b = 2;\n"
    assert bench._code_only(code) == bench._code_only(
        "// header\nint a = 1;   // the first\n\n/* a block\n   comment */\nint b = 2;  \n\n")


def test_code_only_sees_code_changes():
    assert bench._code_only("int a = 1;\n") != bench._code_only("int a = 2;\n")
    assert bench._code_only("f(x); // g(y);\n") != bench._code_only("f(x); g(y);\n")


def test_source_hash_depends_on_the_step_kind():
    hashes = {k: bench.kernel_source_sha(k) for k in ("forward", "split", "backward")}
    assert len(set(hashes.values())) == 3
    assert all(len(h) == 16 for h in hashes.values())


def test_recorded_traffic_matches_the_current_sources():
    # Every committed traffic summary was captured on the kernel sources as they stand.
    for wid in (3, 4, 6, 7, 8):
        traffic = bench.recorded_traffic(wid)
        assert traffic is not None and traffic > 0, f"workload {wid}: traffic summary out of date"
    # Workloads without a committed summary report none.
    assert bench.recorded_traffic(1) is None
