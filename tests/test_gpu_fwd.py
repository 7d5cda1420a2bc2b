"""Forward parity of the CUDA path against the fp64 oracle (GPU)."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL_REL_O, check, check_lse, to64
from causal_gqa_attention_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gq():
    import causal_gqa_attention_fwd_gb300 as g
    g.lib()
    return g


DENSE_CASES = [
    # B, Hq, Hkv, T, D, causal
    (1, 4, 2, 128, 64, True),      # tiny workload
    (1, 2, 1, 200, 128, True),     # ragged T, G = 2
    (2, 3, 3, 300, 64, True),      # MHA, odd row-block count (pairs of row blocks)
    (1, 8, 1, 129, 128, True),     # G = 8, one row past a tile
    (1, 2, 2, 1, 128, True),       # T = 1
    (1, 4, 4, 65, 64, True),       # T = 65
    (1, 6, 2, 333, 128, True),     # G = 3 (odd), ragged
    (1, 4, 2, 200, 128, False),    # non-causal, ragged
    (2, 2, 1, 256, 64, False),     # non-causal, exact tiles
]


@pytest.mark.parametrize("B,Hq,Hkv,T,D,causal", DENSE_CASES)
def test_fwd_dense(gq, B, Hq, Hkv, T, D, causal):
    x = W.dense_inputs(B, Hq, Hkv, T, D, seed=T + D)
    scale = 1.0 / np.sqrt(D)
    o, lse = gq.attn_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), causal=causal, scale=scale)
    assert gq.get_device_status() == 0
    ro, rl = oracle.fwd(to64(x["q"]), to64(x["k"]), to64(x["v"]), causal=causal, scale=scale)
    check("o", o, ro, TOL_REL_O)
    check_lse(lse, rl)


@pytest.mark.parametrize("name", ["tiny", "qwen3_0p6b_layer"])
def test_fwd_workload(gq, name):
    w = W.WORKLOADS[name]
    x = W.make_inputs(w)
    o, lse = gq.attn_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), scale=w.softmax_scale)
    ro, rl = oracle.fwd(to64(x["q"]), to64(x["k"]), to64(x["v"]), scale=w.softmax_scale)
    check("o", o, ro, TOL_REL_O)
    check_lse(lse, rl)


@pytest.mark.parametrize("lens,Hq,Hkv,D,q_std", [
    ([1, 130, 64, 257], 4, 2, 128, 1.0),
    ([5, 300, 129], 3, 3, 64, 4.0),
    ([128, 0, 7], 2, 1, 128, 4.0),
])
def test_fwd_varlen(gq, lens, Hq, Hkv, D, q_std):
    x = W.varlen_inputs(lens, Hq, Hkv, D, seed=sum(lens), q_std=q_std)
    scale = 1.0 / np.sqrt(D)
    cu = x["cu_seqlens"]
    o, lse = gq.attn_varlen_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), cu.cuda(), x["max_seqlen"],
                                scale=scale)
    assert gq.get_device_status() == 0
    ro, rl = oracle.varlen_fwd(to64(x["q"]), to64(x["k"]), to64(x["v"]), cu.numpy(), scale=scale)
    check("o", o, ro, TOL_REL_O)
    check_lse(lse, rl)
