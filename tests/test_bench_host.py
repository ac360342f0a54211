"""Host-side pieces of bench.py that need no GPU."""
import bench


def test_profiled_traffic_follows_the_kernel_sources(monkeypatch):
    # every kernel named in the committed summaries resolves to a byte count or,
    # once its sources differ from the profiled ones, to None
    for k in bench.KERNEL_SOURCES:
        v = bench.profiled_traffic(k)
        assert v is None or (isinstance(v, int) and v > 0)
    monkeypatch.setattr(bench, "sources_digest", lambda kernel: "0" * 16)
    for k in bench.KERNEL_SOURCES:
        assert bench.profiled_traffic(k) is None
    assert bench.profiled_traffic("no_such_kernel") is None


def test_per_token_work_of_the_prefill_workload():
    import workloads as W
    w = W.PREFILL_BF16
    work = bench.per_token_work(w)
    # 16 rows of 128 B in, 2 KiB of e out, the raw id and its projection
    assert work["hash_gather"] == ("bytes", 8 + 16 * 128 + 2 * 1024)
    assert work["kv_gemm"] == ("flops", 2 * 1024 * 2048)
    assert work["stage_b"] == work["kv_gemm"]
    # v fp32, the (s, alpha) row, H read and written in bf16
    assert work["conv"] == ("bytes", 4 * 1024 + 8 + 2 * 2 * 1024)
