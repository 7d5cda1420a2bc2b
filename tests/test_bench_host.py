"""bench.py's host-side legs on CPU: the oracle baseline on every prefill
workload kind (dense groups and packed sequences) and the decode parity leg
(plain, paged and E4M3 caches, rotary queries)."""
import pytest
import torch


@pytest.mark.parametrize("name", ["tiny", "varlen16"])
def test_cpu_baseline_sample_runs(name):
    import bench
    from causal_gqa_attention_fwd_gb300 import workloads as W
    w = W.WORKLOADS[name]
    x = W.make_inputs(w)
    rate, desc, cores, elapsed = bench.oracle_sample(w, x, 0.0)   # one group / one sequence
    assert rate > 0 and cores >= 1 and elapsed > 0
    assert ("packed sequences" in desc) == w.varlen


@pytest.mark.parametrize("kind", ["plain", "paged", "fp8", "rope"])
def test_decode_parity_leg_accepts_the_oracle_itself(kind):
    """The decode parity leg, fed the oracle's own output (rounded to bf16),
    passes; fed a corrupted row, it fails.  Small shapes, so the check runs
    on the CPU in seconds."""
    import numpy as np

    import bench
    import oracle
    from causal_gqa_attention_fwd_gb300 import workloads as W
    w = W.DecodeWorkload("small", B=3, Hq=4, Hkv=2, Tq=1, S=256, D=64, min_len=16, max_len=256,
                         page_size=16 if kind == "paged" else 0, fp8=kind == "fp8", rope=kind == "rope")
    x = W.make_decode_inputs(w, seed=3)
    f = lambda t: t.float().numpy().astype(np.float64)
    ln = x["cache_lens"].numpy()
    if kind == "rope":
        assert x["rope_cs"].shape == (w.S, w.D)
        ro, rlse = oracle.decode_fwd(f(x["q"]), f(x["k_cache"]), f(x["v_cache"]), ln, scale=w.softmax_scale,
                                     rope_cos_sin=x["rope_cs"].double().numpy())
        # the leg must hand the table to the oracle: unrotated queries are far off
        plain, _ = oracle.decode_fwd(f(x["q"]), f(x["k_cache"]), f(x["v_cache"]), ln, scale=w.softmax_scale)
        assert not bench.decode_parity_leg(w, x, torch.from_numpy(plain).to(torch.bfloat16),
                                           torch.from_numpy(rlse).float())["pass"]
    elif kind == "fp8":
        ro, rlse = oracle.fp8_decode_fwd(f(x["q"]), x["k8"].numpy(), x["v8"].numpy(), x["k_scale"], x["v_scale"], ln,
                                         scale=w.softmax_scale)
    elif kind == "paged":
        ro, rlse = oracle.paged_decode_fwd(f(x["q"]), f(x["k_pages"]), f(x["v_pages"]), x["block_table"].numpy(), ln,
                                           scale=w.softmax_scale)
    else:
        ro, rlse = oracle.decode_fwd(f(x["q"]), f(x["k_cache"]), f(x["v_cache"]), ln, scale=w.softmax_scale)
    o = torch.from_numpy(ro).to(torch.bfloat16)
    lse = torch.from_numpy(rlse).float()
    good = bench.decode_parity_leg(w, x, o, lse)
    assert good["pass"] and good["outputs"]["o"]["rel_fro"] < 5e-3
    rows = [int(x["cache_lens"].argmin()), int(x["cache_lens"].argmax())]
    o_bad = o.clone()
    o_bad[rows[1]] += 0.5
    assert not bench.decode_parity_leg(w, x, o_bad, lse)["pass"]
