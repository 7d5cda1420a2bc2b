"""Backward with rotary queries and keys on the GPU against the fp64 oracle
(``oracle.rope_bwd`` / ``oracle.rope_varlen_bwd``: the gradients of
L = sum(dO * O) with respect to the unrotated q, k and v, the rotation taken
at positions 0..T-1, or 0..len-1 in every packed sequence).

The CUDA path takes o and lse from attn_fwd_rope, as a user would, rotates q
and k into f16 copies, runs the backward with f16 Q/K operands and an f16 dS,
and takes dQ and dK back through the rotation.  Cases: D 64 and 128, G 1, 2,
3 and 8, causal and not, ragged lengths across several 128-row tiles, the
long-context layer (B 2, Hq 32, Hkv 8, T 4096, D 128) on sampled groups, and a
ragged packed batch.
"""
import numpy as np
import pytest

import oracle
from parity_util import TOL_REL_GRAD, check, to64
from causal_gqa_attention_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gq():
    import causal_gqa_attention_fwd_gb300 as g
    g.lib()
    oracle.set_threads(0)
    return g


def gpu_rope(gq, x, tab, causal, scale):
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    t = tab.cuda()
    o, lse = gq.attn_fwd_rope(q, k, v, t, causal=causal, scale=scale)
    dq, dk, dv = gq.attn_bwd_rope(q, k, v, o, lse, do, t, causal=causal, scale=scale)
    assert gq.get_device_status() == 0
    return dq.cpu(), dk.cpu(), dv.cpu()


CASES = [
    # B, Hq, Hkv, T, D, causal
    (1, 4, 2, 128, 64, True),
    (2, 2, 1, 333, 128, True),
    (1, 6, 2, 200, 128, True),     # G = 3
    (1, 8, 1, 1000, 128, True),    # G = 8
    (2, 3, 3, 300, 64, True),      # MHA
    (1, 4, 2, 200, 128, False),
    (1, 2, 2, 1, 64, True),        # T = 1
]


@pytest.mark.parametrize("B,Hq,Hkv,T,D,causal", CASES)
def test_bwd_rope_matches_oracle(gq, B, Hq, Hkv, T, D, causal):
    x = W.dense_inputs(B, Hq, Hkv, T, D, seed=T + D + 11)
    tab = W.rope_cos_sin_table(T + 3, D)
    scale = 1.0 / np.sqrt(D)
    dq, dk, dv = gpu_rope(gq, x, tab, causal, scale)
    ref = oracle.rope_bwd(to64(x["q"]), to64(x["k"]), to64(x["v"]), to64(x["do"]), tab.double().numpy(),
                          causal=causal, scale=scale, err_terms=True)
    check("dq", dq, ref["dq"], TOL_REL_GRAD, ref["edq"])
    check("dk", dk, ref["dk"], TOL_REL_GRAD, ref["edk"])
    check("dv", dv, ref["dv"], TOL_REL_GRAD, ref["edv"])


@pytest.fixture(scope="module")
def long_rope(gq):
    w = W.WORKLOADS["long_gqa_t4096"]
    x = W.make_inputs(w)
    tab = W.rope_cos_sin_table(w.T, w.D)
    return w, x, tab, gpu_rope(gq, x, tab, True, w.softmax_scale)


@pytest.mark.parametrize("b,g", [(0, 0), (1, 7)])
def test_bwd_rope_long_gqa_t4096_sampled_group(long_rope, b, g):
    w, x, tab, (dq, dk, dv) = long_rope
    G = w.Hq // w.Hkv
    hs = slice(g * G, (g + 1) * G)
    ref = oracle.rope_bwd(to64(x["q"][b:b + 1, hs]), to64(x["k"][b:b + 1, g:g + 1]), to64(x["v"][b:b + 1, g:g + 1]),
                          to64(x["do"][b:b + 1, hs]), tab.double().numpy(), scale=w.softmax_scale, err_terms=True)
    check("dq", dq[b:b + 1, hs], ref["dq"], TOL_REL_GRAD, ref["edq"])
    check("dk", dk[b:b + 1, g:g + 1], ref["dk"], TOL_REL_GRAD, ref["edk"])
    check("dv", dv[b:b + 1, g:g + 1], ref["dv"], TOL_REL_GRAD, ref["edv"])


@pytest.mark.parametrize("lens,Hq,Hkv,D,q_std", [
    ([1, 130, 64, 257], 4, 2, 128, 1.0),
    ([5, 300, 129], 3, 3, 64, 1.0),
    ([700, 0, 33, 1200], 8, 2, 128, 4.0),
])
def test_varlen_bwd_rope_matches_oracle(gq, lens, Hq, Hkv, D, q_std):
    x = W.varlen_inputs(lens, Hq, Hkv, D, seed=19 + sum(lens), q_std=q_std)
    tab = W.rope_cos_sin_table(max(lens) + 1, D)
    scale = 1.0 / np.sqrt(D)
    cu = x["cu_seqlens"]
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    cud, t = cu.cuda(), tab.cuda()
    o, lse = gq.attn_varlen_fwd_rope(q, k, v, cud, x["max_seqlen"], t, scale=scale)
    dq, dk, dv = gq.attn_varlen_bwd_rope(q, k, v, o, lse, do, cud, x["max_seqlen"], t, scale=scale)
    assert gq.get_device_status() == 0
    ref = oracle.rope_varlen_bwd(to64(x["q"]), to64(x["k"]), to64(x["v"]), to64(x["do"]), cu.numpy(),
                                 tab.double().numpy(), scale=scale, err_terms=True)
    check("dq", dq, ref["dq"], TOL_REL_GRAD, ref["edq"])
    check("dk", dk, ref["dk"], TOL_REL_GRAD, ref["edk"])
    check("dv", dv, ref["dv"], TOL_REL_GRAD, ref["edv"])
