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


def test_every_traced_kernel_name_has_its_work():
    """Each name the per-kernel tracing can assign has an algorithmic amount, so a
    traced interval is never reported without a roofline denominator; the codes
    gather moves the rows in and the codes and scale out (no bf16 e)."""
    import workloads as W
    for w in W.ALL:
        work = bench.per_token_work(w)
        for sets in (bench.NAME_SETS, bench.NAME_SETS_FP8, bench.NAME_SETS_DECODE, bench.NAME_SETS_DECODE_FP8):
            for names in sets.values():
                for n in names:
                    assert n in work, (w.name, n)
    w = W.PREFILL_BF16
    work = bench.per_token_work(w)
    assert work["hash_gather_e4m3"] == ("bytes", 8 + 16 * 128 + 1024 + 4)


def test_reference_arm_generates_its_inputs_once(monkeypatch, capsys):
    """The reference arm times the oracle on a sample per step; the layers'
    tables are generated once per process, not once per step, so the run's
    length follows the step count through the oracle's own work only."""
    import argparse
    import json
    import workloads as W
    calls = []
    real = W.layer_inputs

    def counted(*a, **k):
        calls.append(a[1] if len(a) > 1 else k.get("layer"))
        return real(*a, **k)

    monkeypatch.setattr(W, "layer_inputs", counted)
    monkeypatch.setattr(bench, "_ORACLE_INPUTS", None)
    bench.run_reference(argparse.Namespace(steps=4, warmup=1, gpus=1))
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 4 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert len(calls) == len(W.PREFILL_BF16.layers)
