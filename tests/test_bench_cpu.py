"""The CPU leg of bench.py (the oracle timed on the host): the JSON keys the benchmark
contract asks of cpu_baseline, the single-thread figure on the tiny workload, the
per-workload figures (whole tensors; a row sample of FLUX-2048, extrapolated), and that
timing it leaves the oracle's thread count for later calls as it was."""
import bench
import oracle
from workloads import WORKLOADS


def test_cpu_baseline_keys_and_thread_count():
    before = oracle.num_threads()
    r = bench.cpu_baseline(WORKLOADS["tiny"], seconds=0.3, full_workloads=("tiny",), flux2048_rows=8)
    assert r["kind"] == "oracle" and r["unit"] == "TFLOPS" and r["value"] > 0
    assert r["cores"] == before and "query rows of tiny" in r["sample"]
    assert r["extrapolated_full_s"] > 0
    st = r["single_thread_tiny"]
    assert st["value"] > 0 and st["seconds"] > 0 and st["sample"] == "all rows of tiny, 1 thread"
    assert oracle.num_threads() == before
    full = r["per_workload"]
    assert full["tiny"]["value"] > 0 and full["tiny"]["cores"] == before and "every row of tiny" in full["tiny"]["sample"]
    f2 = full["flux2048"]
    assert f2["value"] > 0 and f2["extrapolated_full_s"] > f2["seconds"] and "8 query rows" in f2["sample"]
