"""The bench's CPU legs (no GPU): the oracle single-threaded and on every core.

Both time the oracle as it stands on bounded samples of a workload; the
all-cores leg gives each thread its own copy of the sample, so its threads
share no arrays, and reports the threads it ran.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    sys.path.insert(0, ROOT)
    import bench
    return bench


def test_all_cores_leg_reports_threads_and_sample():
    bench = _bench()
    from zero_partition_aware_gb300 import workloads as W
    d = bench.cpu_baseline_all_cores(W.WORKLOADS["tiny"], 0.5)
    n = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    assert d["kind"] == "oracle" and d["unit"] == "params/s"
    assert d["cores"] == n and d["value"] > 0 and f"{n} threads" in d["sample"]


def test_sample_passes_over_params_larger_than_the_cap():
    bench = _bench()
    from zero_partition_aware_gb300 import workloads as W
    wl = W.replace(W.WORKLOADS["tiny"], numel=(50, 5000, 20, 30, 4000))
    lay = bench.oracle_sample(wl, 100, skip_larger=True)[0]
    assert list(lay.numel) == [50, 20, 30]
    lay = bench.oracle_sample(wl, 100)[0]
    assert list(lay.numel) == [50]


def test_single_thread_leg():
    bench = _bench()
    from zero_partition_aware_gb300 import workloads as W
    d = bench.cpu_baseline(W.WORKLOADS["tiny"], 0.3)
    assert d["cores"] == 1 and d["value"] > 0 and d["kind"] == "oracle"


def test_traffic_hash_ignores_comments_not_code():
    bench = _bench()
    a = "int f(int x) {\n    return x + 1;  // one\n}\n"
    b = "/* doc\n   more */\nint f(int x) {\n\n    return x + 1;\n}   \n// end\n"
    c = "int f(int x) {\n    return x + 2;\n}\n"
    assert bench.code_only(a) == bench.code_only(b) != bench.code_only(c)
    assert len(bench.kernel_source_hash()) == 16


def test_traffic_hash_follows_the_compile_flags(monkeypatch):
    """The profiled traffic is keyed to the host launch code and the nvcc flags
    too: a changed flag must move the hash."""
    bench = _bench()
    from zero_partition_aware_gb300 import build as zb
    h0 = bench.kernel_source_hash()
    monkeypatch.setattr(zb, "COMMON_FLAGS", zb.COMMON_FLAGS + ["-DZR_SOMETHING"])
    assert bench.kernel_source_hash() != h0
