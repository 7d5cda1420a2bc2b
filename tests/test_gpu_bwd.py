"""Backward parity of the CUDA path against the fp64 oracle (GPU).

The CUDA backward consumes the CUDA forward's O and LSE (as a user would);
the oracle recomputes everything from Q, K, V, dO in fp64.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL_REL_GRAD, check, to64
from causal_gqa_attention_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gq():
    import causal_gqa_attention_fwd_gb300 as g
    g.lib()
    return g


def run_dense(gq, x, causal, scale):
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = gq.attn_fwd(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = gq.attn_bwd(q, k, v, o, lse, do, causal=causal, scale=scale)
    assert gq.get_device_status() == 0
    return dq, dk, dv


DENSE_CASES = [
    # B, Hq, Hkv, T, D, causal
    (1, 4, 2, 128, 64, True),      # tiny workload
    (1, 2, 1, 200, 128, True),     # ragged T, G = 2
    (2, 3, 3, 300, 64, True),      # MHA, ragged
    (1, 8, 1, 129, 128, True),     # G = 8, one row past a tile
    (1, 2, 2, 1, 128, True),       # T = 1
    (1, 4, 4, 65, 64, True),       # T = 65
    (1, 6, 2, 333, 128, True),     # G = 3, ragged
    (1, 4, 2, 200, 128, False),    # non-causal, ragged
    (2, 2, 1, 256, 64, False),     # non-causal, exact tiles
    (1, 2, 1, 512, 128, True),     # several key blocks
]


@pytest.mark.parametrize("B,Hq,Hkv,T,D,causal", DENSE_CASES)
def test_bwd_dense(gq, B, Hq, Hkv, T, D, causal):
    x = W.dense_inputs(B, Hq, Hkv, T, D, seed=1000 + T + D)
    scale = 1.0 / np.sqrt(D)
    dq, dk, dv = run_dense(gq, x, causal, scale)
    ref = oracle.bwd(to64(x["q"]), to64(x["k"]), to64(x["v"]), to64(x["do"]), causal=causal, scale=scale,
                     err_terms=True)
    check("dq", dq, ref["dq"], TOL_REL_GRAD, ref["edq"])
    check("dk", dk, ref["dk"], TOL_REL_GRAD, ref["edk"])
    check("dv", dv, ref["dv"], TOL_REL_GRAD, ref["edv"])


@pytest.mark.parametrize("name", ["tiny", "qwen3_0p6b_layer"])
def test_bwd_workload(gq, name):
    w = W.WORKLOADS[name]
    x = W.make_inputs(w)
    dq, dk, dv = run_dense(gq, x, True, w.softmax_scale)
    ref = oracle.bwd(to64(x["q"]), to64(x["k"]), to64(x["v"]), to64(x["do"]), scale=w.softmax_scale,
                     err_terms=True)
    check("dq", dq, ref["dq"], TOL_REL_GRAD, ref["edq"])
    check("dk", dk, ref["dk"], TOL_REL_GRAD, ref["edk"])
    check("dv", dv, ref["dv"], TOL_REL_GRAD, ref["edv"])


@pytest.mark.parametrize("lens,Hq,Hkv,D,q_std", [
    ([1, 130, 64, 257], 4, 2, 128, 1.0),
    ([5, 300, 129], 3, 3, 64, 4.0),
    ([128, 0, 7], 2, 1, 128, 4.0),
])
def test_bwd_varlen(gq, lens, Hq, Hkv, D, q_std):
    x = W.varlen_inputs(lens, Hq, Hkv, D, seed=7 + sum(lens), q_std=q_std)
    scale = 1.0 / np.sqrt(D)
    cu = x["cu_seqlens"]
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    cud = cu.cuda()
    o, lse = gq.attn_varlen_fwd(q, k, v, cud, x["max_seqlen"], scale=scale)
    dq, dk, dv = gq.attn_varlen_bwd(q, k, v, o, lse, do, cud, x["max_seqlen"], scale=scale)
    assert gq.get_device_status() == 0
    ref = oracle.varlen_bwd(to64(x["q"]), to64(x["k"]), to64(x["v"]), to64(x["do"]), cu.numpy(), scale=scale,
                            err_terms=True)
    check("dq", dq, ref["dq"], TOL_REL_GRAD, ref["edq"])
    check("dk", dk, ref["dk"], TOL_REL_GRAD, ref["edk"])
    check("dv", dv, ref["dv"], TOL_REL_GRAD, ref["edv"])
