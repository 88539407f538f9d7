"""bench.py's roofline `traffic` comes from a committed ncu summary only when that summary
was taken on the current kernel source and on the workload being measured; otherwise the
field is null.  The committed summaries must match the current source."""
import bench


def _summary(tmp_path, workload, digest, traffic="123456"):
    p = tmp_path / "summary.md"
    p.write_text("# summary\n\n"
                 f"- workload: `{workload}`\n"
                 f"- kernel_source_sha256_16: `{digest}`\n"
                 f"- traffic_bytes_per_launch: `{traffic}`\n")
    return str(p)


def test_traffic_read_for_the_same_source_and_workload(tmp_path):
    path = _summary(tmp_path, "llama_32k", bench.kernel_source_digest())
    assert bench.profiled_traffic(path, "llama_32k") == 123456.0


def test_traffic_null_for_another_workload(tmp_path):
    path = _summary(tmp_path, "llama_32k", bench.kernel_source_digest())
    assert bench.profiled_traffic(path, "qwen3_64k") is None


def test_traffic_null_once_the_kernel_source_changed(tmp_path):
    path = _summary(tmp_path, "llama_32k", "0000000000000000")
    assert bench.profiled_traffic(path, "llama_32k") is None


def test_traffic_null_without_a_summary(tmp_path):
    assert bench.profiled_traffic(str(tmp_path / "missing.md"), "llama_32k") is None


def test_committed_summaries_match_the_current_kernel():
    for workload in ("llama_32k", "llama_32k_ragged", "qwen3_64k", "llama_10doc", "batch4_p020"):
        assert bench.profiled_traffic(bench.profile_summary(workload), workload) is not None, workload
