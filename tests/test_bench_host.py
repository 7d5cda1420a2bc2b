"""bench.py's host-side legs on CPU: the oracle baseline on every prefill
workload kind (dense groups and packed sequences)."""
import pytest


@pytest.mark.parametrize("name", ["tiny", "varlen16"])
def test_cpu_baseline_sample_runs(name):
    import bench
    from causal_gqa_attention_fwd_gb300 import workloads as W
    w = W.WORKLOADS[name]
    x = W.make_inputs(w)
    rate, desc, cores, elapsed = bench.oracle_sample(w, x, 0.0)   # one group / one sequence
    assert rate > 0 and cores >= 1 and elapsed > 0
    assert ("packed sequences" in desc) == w.varlen
