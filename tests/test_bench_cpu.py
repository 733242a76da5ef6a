"""The CPU leg of bench.py (the oracle timed on the host): the JSON keys the benchmark
contract asks of cpu_baseline, the single-thread figure on the tiny workload, and that
timing it leaves the oracle's thread count for later calls as it was."""
import bench
import oracle
from workloads import WORKLOADS


def test_cpu_baseline_keys_and_thread_count():
    before = oracle.num_threads()
    r = bench.cpu_baseline(WORKLOADS["tiny"], seconds=0.3)
    assert r["kind"] == "oracle" and r["unit"] == "TFLOPS" and r["value"] > 0
    assert r["cores"] == before and "query rows of tiny" in r["sample"]
    assert r["extrapolated_full_s"] > 0
    st = r["single_thread_tiny"]
    assert st["value"] > 0 and st["seconds"] > 0 and st["sample"] == "all rows of tiny, 1 thread"
    assert oracle.num_threads() == before
